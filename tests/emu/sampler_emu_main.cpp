// Runs pkv_seeded_sample's two kernels (sample_chunk_kernel, then
// sample_finish_kernel) on the CPU emulation of CUDA.  The kernels' source is
// the library's sampler.cu up to the end of its namespace, included below as
// "sampler_dev.inc" (written by the test).  Input and output are raw files:
//   in:  int32 B, V, num_slots, ext; fp32 logits[B*V]; int32 slots[B],
//        active[B]; uint64 seeds[S]; int64 steps[S]; fp32 temperature[S];
//        int32 top_k[S]; fp32 top_p[S]; then, when ext != 0 (the further
//        settings of pkv_seeded_sample_ext): fp32 min_p[S], rep_penalty[S];
//        int32 rep_window[S], hist_cap, history[S*hist_cap], hist_len[S],
//        advance
//   out: int32 out_tok[B], out_kind[B], err; when ext != 0 also fp32
//        logprob_raw[B], logprob_proc[B]; int32 hist_len[S],
//        history[S*hist_cap]; int64 steps[S]
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "sampler_dev.inc"

template <class T>
static void rd(FILE *f, std::vector<T> &v, size_t n) {
  v.resize(n);
  if (fread(v.data(), sizeof(T), n, f) != n) {
    fprintf(stderr, "short input\n");
    exit(2);
  }
}

int main(int argc, char **argv) {
  if (argc != 3) return 2;
  FILE *f = fopen(argv[1], "rb");
  if (!f) return 2;
  int32_t hdr[4];
  if (fread(hdr, sizeof(int32_t), 4, f) != 4) return 2;
  const int B = hdr[0], V = hdr[1], S = hdr[2], ext = hdr[3];
  std::vector<float> logits, temp, top_p;
  std::vector<int32_t> slots, active, top_k;
  std::vector<uint64_t> seeds;
  std::vector<int64_t> steps;
  rd(f, logits, (size_t)B * V);
  rd(f, slots, B);
  rd(f, active, B);
  rd(f, seeds, S);
  rd(f, steps, S);
  rd(f, temp, S);
  rd(f, top_k, S);
  rd(f, top_p, S);
  std::vector<float> min_p, pen, lp_raw(B, 7.0f), lp_proc(B, 7.0f);
  std::vector<int32_t> window, history, hist_len, misc;
  int cap = 1, advance = 0;
  if (ext) {
    rd(f, min_p, S);
    rd(f, pen, S);
    rd(f, window, S);
    rd(f, misc, 1);
    cap = misc[0];
    rd(f, history, (size_t)S * cap);
    rd(f, hist_len, S);
    rd(f, misc, 1);
    advance = misc[0];
  }
  fclose(f);

  using namespace pkv;
  std::vector<int32_t> out_tok(B, -1), out_kind(B, -1);
  int32_t err = 0;
  SampleArgs a{};
  a.logits = logits.data();
  a.row_stride = V;
  a.batch = B;
  a.vocab = V;
  a.nch = chunks_for(V);
  a.slots = slots.data();
  a.active = active.data();
  a.num_slots = S;
  a.seeds = seeds.data();
  a.steps = steps.data();
  a.temperature = temp.data();
  a.top_k = top_k.data();
  a.top_p = top_p.data();
  a.salt = 0;
  a.advance = advance;
  a.out_tok = out_tok.data();
  a.out_kind = out_kind.data();
  const size_t rec_bytes = align_up((size_t)B * a.nch * sizeof(ChunkRec), 256);
  const size_t bytes = rec_bytes + align_up((size_t)B * a.nch * (CHUNK / 8), 256);
  void *ws = aligned_alloc(256, bytes);
  memset(ws, 0xAB, bytes);  // not zeroed: the kernels must not read what they did not write
  a.recs = static_cast<ChunkRec *>(ws);
  if (ext) {
    a.min_p = min_p.data();
    a.rep_penalty = pen.data();
    a.rep_window = window.data();
    a.history = history.data();
    a.hist_len = hist_len.data();
    a.hist_cap = cap;
    a.lp_raw = lp_raw.data();
    a.lp_proc = lp_proc.data();
    a.pbits = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(ws) + rec_bytes);
  }
  a.err = &err;
  // the second CTA per chunk for the normaliser: on unless EMU_ZSPLIT=0
  const char *zs = std::getenv("EMU_ZSPLIT");
  a.zsplit = (zs != nullptr && zs[0] == '0') ? 0 : 1;
  const char *sg = std::getenv("EMU_SINGLE");
  if (a.nch == 1 && !(sg != nullptr && sg[0] == '0')) {
    // one chunk a row: the host launches the single-CTA kernel (EMU_SINGLE=0:
    // the two kernels instead, to compare the two)
    emu_launch(sample_single_kernel, dim3(B), SB, a);
  } else {
    emu_launch(sample_chunk_kernel, dim3(a.nch, B * (1 + a.zsplit)), SB, a);
    emu_launch(sample_finish_kernel, dim3(B), SB, a);
  }
  free(ws);

  FILE *o = fopen(argv[2], "wb");
  if (!o) return 2;
  fwrite(out_tok.data(), sizeof(int32_t), B, o);
  fwrite(out_kind.data(), sizeof(int32_t), B, o);
  fwrite(&err, sizeof(int32_t), 1, o);
  if (ext) {
    fwrite(lp_raw.data(), sizeof(float), B, o);
    fwrite(lp_proc.data(), sizeof(float), B, o);
    fwrite(hist_len.data(), sizeof(int32_t), S, o);
    fwrite(history.data(), sizeof(int32_t), (size_t)S * cap, o);
    fwrite(steps.data(), sizeof(int64_t), S, o);
  }
  fclose(o);
  return 0;
}
