"""The seeded input generator: published SplitMix64 values, determinism, shapes, needles."""
import numpy as np
import pytest
import torch

from synthetic import configs, generator as gen


def test_splitmix64_known_values():
    # Reference outputs of SplitMix64 seeded with state 0 (first three next() calls),
    # as printed with the published algorithm (Vigna's splitmix64.c test vector).
    assert gen.splitmix64_int(0, 0) == 0xE220A8397B1DCDAF
    assert gen.splitmix64_int(0, 1) == 0x6E789E6AA1B965F4
    assert gen.splitmix64_int(0, 2) == 0x06C45D188009454F


@pytest.mark.parametrize("key", [0, 12345, (1 << 64) - 1, gen.stream_key(7, 3, 2)])
def test_splitmix64_torch_matches_int(key):
    idx = [0, 1, 2, 1000, (1 << 31) + 5, (1 << 40) + 17]
    got = gen.splitmix64_torch(key, torch.tensor(idx, dtype=torch.int64)).tolist()
    want = [gen._to_i64(gen.splitmix64_int(key, i)) for i in idx]
    assert got == want


def test_normal_table_quantiles():
    t = gen.normal_table("cpu").double().numpy()
    assert t.shape == (65536,)
    assert np.all(np.diff(t) > 0)
    assert np.allclose(t, -t[::-1], atol=1e-6)           # symmetric quantiles
    assert abs(t.mean()) < 1e-6 and abs(t.var() - 1.0) < 2e-3


def test_normal_stream_is_counter_based():
    key = gen.stream_key(1, 2, 3)
    full = gen.normal_f32(key, 5000, "cpu")
    part = gen.normal_f32(key, 1000, "cpu", start=2000)
    assert torch.equal(full[2000:3000], part)
    assert torch.equal(full, gen.normal_f32(key, 5000, "cpu"))
    assert abs(float(full.mean())) < 0.06 and abs(float(full.var()) - 1) < 0.08


def test_uniform_scale_exact_range():
    s = gen.uniform_scale_f32(gen.stream_key(9), 4096, 0.5, 2.0, "cpu")
    assert float(s.min()) >= 0.5 and float(s.max()) < 2.0
    assert abs(float(s.mean()) - 1.25) < 0.03


def test_tiny_workload_shapes_and_planted_chunk():
    wl = configs.tiny()
    q, k, v, spans = gen.make_all_layers(wl, "cpu")
    assert q[0].shape == (1, 8, 4, 64) and q[0].dtype == torch.float32
    assert k[0].shape == (512, 2, 64) and v[0].shape == (512, 2, 64)
    (s, e), = spans[0][0]
    assert e - s == wl.c and s % wl.c == 0 and e <= 512 - wl.w
    # the planted keys equal the needle vector of each KV head
    vec = gen.needle_vectors(wl, q[0])
    for h in range(2):
        assert np.allclose(k[0][s:e, h].double().numpy(), vec[0, h].astype(np.float32), atol=0)


def test_spans_non_overlapping_and_kept_across_layers():
    wl = configs.llama_model().with_params(seqlens=(4096,), n_layers=4)
    spans = gen.needle_spans(wl)
    for layer in spans:
        (sp,) = layer
        assert len(sp) == 20
        sp = sorted(sp)
        for (a, b), (c2, d2) in zip(sp, sp[1:]):
            assert b <= c2
        for a, b in sp:
            assert 5 <= b - a <= 40 and b <= 4096 - wl.w
    for l0, l1 in zip(spans, spans[1:]):
        assert len(set(l0[0]) & set(l1[0])) == 16


def test_ragged_seqlens_in_range():
    wl = configs.mistral_ragged()
    assert len(wl.seqlens) == 16 and all(4096 <= t <= 16384 for t in wl.seqlens)
    assert wl.cu_seqlens[-1] == sum(wl.seqlens)


def test_channel_scale_applied_per_channel():
    wl = configs.llama_layer().with_params(seqlens=(2048,))
    k = gen.gen_kv_raw(wl, 0, gen.TENSOR_K, "cpu").float()
    std = k.std(dim=0)                       # [Hkv, d]
    assert float(std.min()) > 0.4 and float(std.max()) < 2.2
    assert float(std.max() / std.min()) > 2.0
