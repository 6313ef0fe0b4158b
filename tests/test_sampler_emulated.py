"""The sampler kernels' CUDA source, run on the CPU.

tests/emu/cuda_emu.h emulates the CUDA primitives the sampler uses (block
barriers, warp shuffles / ballots / reductions, atomics) with one std::thread
per CUDA thread; the library's csrc/sampler.cu is compiled against it with
address and undefined-behaviour sanitizers (bounds, alignment) and run on
seeded inputs.  The sampled tokens must equal the oracle's except at
near-ties, as on the GPU.  Lanes of a warp never run in lockstep here, so a
warp-synchronous assumption in the kernels shows up as a wrong token, and an
out-of-bounds or misaligned access stops the run.  No GPU is needed; this is
a check of the kernels' logic, not a fallback (nothing in the library calls
it)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NEAR = 1e-6


@pytest.fixture(scope="module")
def emu_binary(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("sampler_emu")
    src = open(os.path.join(ROOT, "paged_kv_decode_pages_gb300", "csrc", "sampler.cu")).read()
    end = src.index("}  // namespace pkv") + len("}  // namespace pkv")
    (d / "sampler_dev.inc").write_text(src[:end] + "\n")
    exe = d / "sampler_emu"
    cmd = [gxx, "-std=c++20", "-O1", "-g", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=all", "-ffp-contract=off",
           "-I", os.path.join(ROOT, "tests", "emu"), "-I", os.path.join(ROOT, "include"),
           "-I", str(d), os.path.join(ROOT, "tests", "emu", "sampler_emu_main.cpp"),
           "-o", str(exe), "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True)
    return exe


def _run(exe, tmp_path, x, slots, active, seeds, steps, temp, top_k, top_p):
    B, V = x.shape
    S = seeds.shape[0]
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        np.array([B, V, S], np.int32).tofile(f)
        for arr, dt in ((x, np.float32), (slots, np.int32), (active, np.int32), (seeds, np.uint64),
                        (steps, np.int64), (temp, np.float32), (top_k, np.int32),
                        (top_p, np.float32)):
            np.ascontiguousarray(arr, dtype=dt).tofile(f)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0")
    r = subprocess.run([str(exe), str(inp), str(out)], capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = np.fromfile(out, np.int32)
    return res[:B], res[B:2 * B], int(res[2 * B])


CASES = [
    # B, V, std, T, k, p, dist
    (3, 1024, 2.0, 0.0, 0, 1.0, "normal"),        # greedy
    (3, 6561, 3.0, 1.0, 25, 0.8, "normal"),       # top-k 25 + top-p, one chunk
    (3, 20000, 1.0, 1.0, 0, 1.0, "normal"),       # keep everything (fp32 Gumbel scores)
    (3, 20000, 1.0, 5.0, 0, 0.95, "normal"),      # top-p crossing past 512 tokens
    (3, 40000, 1.0, 1.0, 200, 0.99, "normal"),    # top-k above the per-chunk candidates
    (3, 40000, 1.0, 1.0, 300, 0.99, "conc"),      # one chunk holds the top-k
    (3, 40000, 1.0, 1.0, 513, 1.0, "normal"),     # general path: top-k > 512
    (2, 151936, 4.0, 0.7, 0, 0.95, "normal"),     # long-context sampler
    (2, 151936, 1.0, 0.5, 0, 0.95, "conc"),       # one chunk holds the top-p set
]


@pytest.mark.parametrize("B,V,std,T,k,p,dist", CASES)
def test_emulated_sampler_matches_oracle(emu_binary, tmp_path, B, V, std, T, k, p, dist):
    rng = np.random.default_rng(V + k)
    x = rng.normal(0, std, (B, V)).astype(np.float32)
    if dist == "conc":
        x[:, :8192] += np.float32(6.0)
    x[0, 3 % V] = -np.inf  # a masked token
    B1 = B + 1  # plus one padding row
    x = np.concatenate([x, np.zeros((1, V), np.float32)])
    slots = np.arange(1, B1 + 1, dtype=np.int32)
    slots[-1] = 0
    active = np.ones(B1, np.int32)
    active[-1] = 0
    S = B1 + 1
    seeds = (np.arange(S, dtype=np.uint64) + np.uint64(977))
    steps = np.full(S, 3, np.int64)
    temp = np.full(S, T, np.float32)
    top_k = np.full(S, k, np.int32)
    top_p = np.full(S, p, np.float32)
    got, kind, err = _run(emu_binary, tmp_path, x, slots, active, seeds, steps, temp, top_k, top_p)
    want, wkind, info, _ = oracle.seeded_sample(x, slots, active, seeds, steps.copy(), temp,
                                                   top_k, top_p, advance=False)
    assert err & ~0x10 == 0  # only the logits bit (the -inf token) may be set
    near = (info["top2_gap_rel"] < NEAR) | (info["member_margin"] < NEAR)
    mism = got != want
    assert not np.any(mism & ~near), (np.nonzero(mism & ~near), got, want)
    assert got[-1] == 0 and kind[-1] == 0
