"""bench.py's algorithmic amounts, the numerators of its throughput and roofline figures (CPU only).

Per step the scoring reads K of every scoring layer once (T_total * Hkv * d * elt a group) and does
2 * w * G * T_total * Hkv * d flops; the finalisation reads one 16-bit bin per (chunk, window row,
KV head) a group; the gather reads and writes the kept K and V rows of every layer.  The figures
below are those amounts written out by hand for the two bench workloads, with the kept counts the
capacity rule gives (min(T, floor(L_max / c) * c + min(w, T)) rows a head).
"""
import numpy as np
import pytest
import torch

import bench
from synthetic import configs

PEAKS = {"hbm_gbs": 6770.1, "bf16_tflops": 1917.0, "bf16_tflops_sustained": 1713.4}


def _full_counts(wl):
    groups = -(-wl.n_layers // wl.n_reuse)
    cnt = np.zeros((groups, wl.B, wl.Hkv), dtype=np.int32)
    for b, T in enumerate(wl.seqlens):
        cnt[:, b, :] = min(T, (wl.L_max // wl.c) * wl.c + min(wl.w, T))
    return torch.from_numpy(cnt)


@pytest.mark.parametrize("head", [True, False])
def test_llama3_32k_amounts(monkeypatch, head):
    wl = configs.llama_model()
    assert (wl.n_layers, wl.n_reuse, wl.T_total, wl.Hkv, wl.d, wl.w, wl.G, wl.c) == (32, 2, 32768, 8, 128, 32, 4, 10)
    counts = _full_counts(wl)
    assert int(counts[0, 0, 0]) == 655 * 10 + 32
    monkeypatch.setattr(bench, "head_path", lambda wl, groups: head)
    ms = {"score": 0.2, "finalize": 0.05, "gather": 0.3}
    (score, fin, gather), _ = bench.phase_rooflines(wl, counts, ms, PEAKS, "measured", 1)
    assert score["algorithmic_bytes"] == 16 * 32768 * 8 * 128 * 2                 # 1.074 GB
    assert score["bound"] == "hbm"                  # 137 GF take 80 us at the tensor roof, 1.07 GB 159 us
    assert fin["algorithmic_bytes"] == 16 * 3277 * 8 * 32 * 4 * 2                  # 107 MB
    assert fin["kernel"] == ("head_kernel" if head else "finalize_kernel")
    assert gather["algorithmic_bytes"] == 4 * 32 * 8 * 6582 * 128 * 2              # 1.725 GB
    for r in (score, fin, gather):
        assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / (ms[r["phase"]] * 1e-3) / 1e9, abs=0.006)
        assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"], abs=1e-4)
    q_bytes = 16 * 32 * 32 * 128 * 2
    assert bench.algorithmic_bytes(wl, counts) == score["algorithmic_bytes"] + q_bytes + gather["algorithmic_bytes"]


def test_qwen2_128k_scoring_is_tensor_bound(monkeypatch):
    wl = configs.qwen_128k()
    assert (wl.n_layers, wl.n_reuse, wl.T_total, wl.Hkv, wl.w, wl.G, wl.c) == (28, 2, 131072, 4, 64, 7, 10)
    monkeypatch.setattr(bench, "head_path", lambda wl, groups: False)
    ms = {"score": 0.8, "finalize": 0.1, "gather": 0.25}
    (score, fin, gather), _ = bench.phase_rooflines(wl, _full_counts(wl), ms, PEAKS, "measured", 1)
    flops = 2.0 * 14 * 64 * 7 * 131072 * 4 * 128                                   # 842 GF
    assert score["bound"] == "tensor" and score["algorithmic_flops"] == flops
    assert flops / (PEAKS["bf16_tflops_sustained"] * 1e12) > score["algorithmic_bytes"] / (PEAKS["hbm_gbs"] * 1e9)
    assert score["achieved"] == pytest.approx(flops / 0.8e-3 / 1e12, abs=0.006)
    assert score["frac"] == pytest.approx(score["achieved"] / PEAKS["bf16_tflops_sustained"], abs=1e-4)
    assert fin["kernel"] == "finalize_kernel"
    assert fin["algorithmic_bytes"] == 14 * 13108 * 4 * 64 * 7 * 2                 # 0.66 GB
    kept = (131072 * 10 // 100) // 10 * 10 + 64
    # 1.51 GB at full capacity; the bench's own counts are smaller where a selected chunk overlaps the
    # recent window (1.48 GB measured)
    assert gather["algorithmic_bytes"] == 4 * 28 * 4 * kept * 128 * 2


def test_portable_path_is_reported_against_hbm(monkeypatch):
    wl = configs.llama_model().with_params(n_layers=2)
    monkeypatch.setattr(bench, "head_path", lambda wl, groups: False)
    ms = {"score": 1.0, "finalize": 0.1, "gather": 0.1}
    score = bench.phase_rooflines(wl, _full_counts(wl), ms, PEAKS, "measured", 0)[0][0]
    assert score["kernel"] == "score_simt_kernel" and score["bound"] == "hbm"


@pytest.mark.parametrize("rate,bound", [(10.0e12, "tensor"), (5.0e12, "sfu")])
def test_exponential_roof_of_the_128k_scoring(monkeypatch, rate, bound):
    # one base-2 exponential per logit: 14 scoring layers x 448 window rows x 131072 keys x 4 KV heads
    # (3.29 G).  At 10 T exp/s they take 329 us, under the 491 us of the sustained tensor roof; at
    # 5 T exp/s they take 658 us and the exponential unit binds.
    wl = configs.qwen_128k()
    monkeypatch.setattr(bench, "head_path", lambda wl, groups: False)
    ms = {"score": 0.8, "finalize": 0.1, "gather": 0.25}
    (score, _, _), every = bench.phase_rooflines(wl, _full_counts(wl), ms, PEAKS, "measured", 1,
                                                 {"exp_per_s": rate})
    exps = 14 * 448 * 131072 * 4
    sfu = next(r for r in every if r["bound"] == "sfu")
    assert sfu["algorithmic_exps"] == exps and sfu["unit"] == "Gexp/s"
    assert sfu["ideal_ms"] == pytest.approx(exps / rate * 1e3, abs=1e-5)
    assert sfu["achieved"] == pytest.approx(exps / 0.8e-3 / 1e9, abs=0.006)
    assert sfu["frac"] == pytest.approx(exps / 0.8e-3 / rate, abs=1e-4)
    assert [r["bound"] for r in every] == ["hbm", "tensor", "sfu"]
    assert score["bound"] == bound and score["ideal_ms"] == max(r["ideal_ms"] for r in every)


def test_job_rate_counts_every_rank():
    assert bench.job_rate(100.0, 4, 2.0) == pytest.approx(200000.0)


def test_cpulist_parsing():
    # the host CPUs local to the GPU come from a Linux cpulist in sysfs
    import bench
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("72-143") == set(range(72, 144))
    assert bench.parse_cpulist("") == set()


def test_tail_case_keeps_the_prefill_prefix_and_ratio():
    import bench
    from synthetic import configs
    base = configs.llama_model()
    wl, n_prev, L_tail = bench.tail_case(base, 4096)
    kept = base.L_max // base.c * base.c + base.w            # k c + w positions of a prefill pass
    assert n_prev == [min(T, kept) for T in base.seqlens] and wl.seqlens == tuple(x + 4096 for x in n_prev)
    assert L_tail == base.L_max * 4096 // max(base.seqlens) and wl.B == base.B and wl.n_layers == base.n_layers
    rag = configs.mistral_ragged()
    wl, n_prev, L_tail = bench.tail_case(rag, 100)
    assert all(p <= T for p, T in zip(n_prev, rag.seqlens)) and L_tail == rag.c    # one chunk at least
    assert wl.cu_seqlens[-1] == sum(n_prev) + 100 * rag.B
