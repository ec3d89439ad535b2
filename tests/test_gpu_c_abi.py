"""The library from a plain C caller.

tests/c_abi/compress_c.c uses nothing but include/chunkkv.h, the CUDA runtime and
the in-tree libchunkkv.so: it allocates its own device buffers, runs
chunkkv_compress_layers (ChunkKV §4.2 Algorithm 2 around §4.1 Algorithm 1) and
writes the outputs to files.  This test compiles it with the system C compiler,
feeds it a seeded ragged batch and holds its outputs to the CPU oracle under the
usual rules (tests/parity.py).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from parity import check_gather, check_indices, check_scores, f64
from synthetic import configs, generator as gen
from synthetic.generator import NeedleSpec

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "chunk_level_kv_gb300")


def _raw(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()


def test_compress_layers_from_c(tmp_path):
    import chunk_level_kv_gb300  # noqa: F401  (fails loudly if the library was not built)
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "a C compiler is needed to build the C caller"
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "compress_c")
    subprocess.run([cc, "-std=c99", "-O2", "-Wall", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi", "compress_c.c"),
                    f"-L{PKG}", "-l:libchunkkv.so", f"-L{os.path.join(cuda, 'lib64')}", "-lcudart",
                    f"-Wl,-rpath,{PKG}", "-o", exe], check=True, capture_output=True)

    seqlens = (1000, 333, 2500)
    wl = configs.mistral_ragged().with_params(seqlens=seqlens, B=len(seqlens), n_layers=2, n_reuse=2, L_max=300,
                                              needles=NeedleSpec(kind="none"), name="c_caller")
    qs, ks, vs, _ = gen.make_all_layers(wl, "cpu")
    cu = wl.cu_seqlens
    with open(tmp_path / "meta.txt", "w") as f:
        f.write(f"{wl.B} {wl.Hq} {wl.Hkv} {wl.d} {wl.w} {wl.c} {wl.L_max} {wl.n_layers} {wl.n_reuse} 1\n")
        f.write(" ".join(str(x) for x in cu) + "\n")
    for layer in range(wl.n_layers):
        if qs[layer] is not None:
            _raw(qs[layer]).tofile(tmp_path / f"q{layer}.bin")
        _raw(ks[layer]).tofile(tmp_path / f"k{layer}.bin")
        _raw(vs[layer]).tofile(tmp_path / f"v{layer}.bin")
    run = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr

    n_cap, c_max = (int(x) for x in open(tmp_path / "out_meta.txt").read().split())
    groups = -(-wl.n_layers // wl.n_reuse)
    counts = np.fromfile(tmp_path / "counts.bin", dtype=np.int32).reshape(groups, wl.B, wl.Hkv)
    indices = np.fromfile(tmp_path / "indices.bin", dtype=np.int32).reshape(groups, wl.B, wl.Hkv, max(n_cap, 1))
    scores = np.fromfile(tmp_path / "scores.bin", dtype=np.float32).reshape(groups, wl.B, wl.Hkv, max(c_max, 1))
    ref = oracle.compress_layers([f64(x) if x is not None else None for x in qs], [f64(x) for x in ks],
                                 [f64(x) for x in vs], cu, wl.Hq, wl.Hkv, wl.w, wl.c, wl.L_max, wl.n_reuse,
                                 want_kv=False)
    for b, T in enumerate(seqlens):
        for h in range(wl.Hkv):
            A = ref["scores"][0][b][h]
            what = f"C caller sequence {b} head {h}"
            check_scores(scores[0, b, h], A, what)
            n = int(counts[0, b, h])
            got = indices[0, b, h, :n]
            check_indices(got, A, T, wl.c, wl.w, wl.L_max, what)
            for layer in range(wl.n_layers):
                ko = np.fromfile(tmp_path / f"ko{layer}.bin", dtype=np.int16).reshape(wl.B, wl.Hkv, n_cap, wl.d)
                vo = np.fromfile(tmp_path / f"vo{layer}.bin", dtype=np.int16).reshape(wl.B, wl.Hkv, n_cap, wl.d)
                kl = torch.from_numpy(ko[b, h, :n].copy()).view(torch.bfloat16)
                vl = torch.from_numpy(vo[b, h, :n].copy()).view(torch.bfloat16)
                check_gather(kl, ks[layer][cu[b]:cu[b + 1], h], got, f"{what} layer {layer} K'")
                check_gather(vl, vs[layer][cu[b]:cu[b + 1], h], got, f"{what} layer {layer} V'")
