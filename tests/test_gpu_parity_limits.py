"""CUDA library vs CPU oracle at the limits of its kernel instances and launch splits (needs a GB300;
calls go through the C-ABI).

Each case runs a path that the workloads of test_gpu_parity.py do not reach: a scoring instance
(c = 4 with w*G = 256 at compile time, c = 8), the gather for rows that are not a power-of-two
number of 16-byte vectors, every selection instance at its chunk limit and one above, the fused
head kernel's 16-key instance, scoring / packing / gather launches split over many layers, host
window queries, the outputs the header leaves unwritten, and rows whose values outgrow their
first-tile reference (the scoring kernel's rescale).
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from synthetic import configs, generator as gen
from synthetic.generator import NeedleSpec
from test_gpu_parity import run_and_check

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def ckv():
    import chunk_level_kv_gb300 as m     # fails loudly if the library was not built
    return m


@pytest.mark.parametrize("T,c,w,Hq,Hkv,L_max", [
    (3001, 4, 64, 32, 8, 300),       # c = 4, window rows 256 (the compile-time w*G = 256 instance)
    (2050, 8, 32, 32, 8, 256),       # c = 8, window rows 128
])
def test_more_tensor_core_instances(ckv, T, c, w, Hq, Hkv, L_max):
    wl = configs.llama_layer().with_params(seqlens=(T,), c=c, w=w, Hq=Hq, Hkv=Hkv, L_max=L_max,
                                           name=f"bf16_T{T}_c{c}_w{w}_G{Hq // Hkv}")
    p, keep = ckv.make_params(cu_seqlens=wl.cu_seqlens, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, w=wl.w, c=wl.c,
                              L_max=wl.L_max, dtype=torch.bfloat16)
    assert ckv.chunkkv_score_path(p) == 1
    run_and_check(ckv, wl)


# d = 96 bf16 and d = 80 f32 give 12 and 20 sixteen-byte vectors a row
@pytest.mark.parametrize("d,dtype", [(96, "bf16"), (80, "f32")])
def test_gather_rows_of_any_vector_count(ckv, d, dtype):
    wl = configs.llama_layer().with_params(seqlens=(900,), d=d, dtype=dtype, Hq=8, Hkv=2, w=8, L_max=100,
                                           name=f"d{d}_{dtype}")
    run_and_check(ckv, wl)


@pytest.mark.parametrize("w", [32, 48])
def test_more_layers_than_one_launch_takes(ckv, w):
    # 70 layers scored one by one (N_reuse = 1): 70 reuse groups take three scoring launches of at most
    # 32 groups, 70 layers take two gather launches of at most 64, and with w = 48 (window rows packed
    # first) two packing launches of at most 64 layers; the groups on both sides of every boundary are
    # checked against the oracle, with the K' and V' of their layers
    wl = configs.llama_model().with_params(seqlens=(700, 301), B=2, Hq=8, Hkv=2, w=w, n_layers=70, n_reuse=1,
                                           L_max=200, needles=NeedleSpec(kind="none"), name=f"layers70_w{w}")
    n0 = ckv.chunkkv_launch_count()
    run_and_check(ckv, wl, layers_to_check=[0, 31, 32, 63, 64, 69])
    packs = 0 if 128 % w == 0 else 2
    assert ckv.chunkkv_launch_count() - n0 == packs + 3 + 3 + 2     # pack, score, lse / finalize / select, gather


def test_head_kernel_with_more_than_4096_chunks(ckv):
    # one wave of 15 sequences x 8 KV heads = 120 heads whose longest sequence has 4334 chunks of 3
    # tokens: the fused head kernel with 16 selection keys a thread (three launches per call)
    rng = np.random.default_rng(77)
    seqlens = (13000,) + tuple(int(x) for x in rng.integers(0, 3000, size=14))
    wl = configs.mistral_ragged().with_params(seqlens=seqlens, B=len(seqlens), c=3, L_max=900, n_layers=2,
                                              n_reuse=2, needles=NeedleSpec(kind="none"), name="head_c3_4334")
    n0 = ckv.chunkkv_launch_count()
    run_and_check(ckv, wl, seqs=[0, 1, 14])
    assert ckv.chunkkv_launch_count() - n0 == 3                    # score, head_kernel, gather


@pytest.mark.parametrize("n_layers", [6, 2])
def test_outputs_beyond_counts_are_left_unwritten(ckv, n_layers):
    # rows at or beyond counts[b][h] of indices / k_out / v_out and chunk scores at or beyond C_b are left
    # unwritten: sentinels placed there survive a call, with the fused head kernel (6 layers: 120 heads)
    # and with separate log-sum-exp, finalisation and selection launches (2 layers: 40 heads)
    seqlens = (3000, 77, 5, 4096, 0)
    wl = configs.mistral_ragged().with_params(seqlens=seqlens, B=len(seqlens), n_layers=n_layers, n_reuse=2,
                                              L_max=600, needles=NeedleSpec(kind="none"), name="unwritten")
    qs, ks, vs, _ = gen.make_all_layers(wl, DEV)
    p, keep = ckv.params_for(qs[0], ks[0], wl.cu_seqlens, Hkv=wl.Hkv, w=wl.w, c=wl.c, L_max=wl.L_max)
    n_cap, C_max = ckv.chunkkv_out_capacity(p)
    groups = -(-wl.n_layers // wl.n_reuse)
    ko = [torch.full((wl.B, wl.Hkv, n_cap, wl.d), -3.5, dtype=ks[0].dtype, device=DEV) for _ in range(wl.n_layers)]
    vo = [torch.full_like(x, 7.25) for x in ko]
    idx = torch.full((groups, wl.B, wl.Hkv, n_cap), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((groups, wl.B, wl.Hkv), -1, dtype=torch.int32, device=DEV)
    sc = torch.full((groups, wl.B, wl.Hkv, C_max), float("nan"), device=DEV)
    ws = torch.zeros(ckv.chunkkv_workspace_size(p, wl.n_layers, wl.n_reuse), dtype=torch.uint8, device=DEV)
    ckv.chunkkv_compress_layers(p, wl.n_reuse, qs, ks, vs, ko, vo, idx, cnt, sc, ws)
    torch.cuda.synchronize()
    del keep
    assert ckv.chunkkv_status_check(ws) == 0
    idx, cnt, sc = idx.cpu(), cnt.cpu(), sc.cpu()
    for g in range(groups):
        for b, T in enumerate(seqlens):
            C = -(-T // wl.c)
            for h in range(wl.Hkv):
                n = int(cnt[g, b, h])
                assert 0 <= n <= n_cap and (n > 0) == (T > 0)
                assert (idx[g, b, h, n:] == -7).all() and (idx[g, b, h, :n] >= 0).all()
                assert not torch.isnan(sc[g, b, h, :C]).any() and torch.isnan(sc[g, b, h, C:]).all()
                for layer in range(g * wl.n_reuse, min((g + 1) * wl.n_reuse, wl.n_layers)):
                    assert (ko[layer][b, h, n:] == -3.5).all() and (vo[layer][b, h, n:] == 7.25).all()


@pytest.mark.parametrize("many_heads,C_max", [
    (False, 4096), (False, 4097), (False, 13312), (False, 13313), (False, 16384), (False, 16385), (False, 32768),
    (False, 32769),
    (True, 2048), (True, 2049), (True, 4096), (True, 4097), (True, 6144), (True, 6145)])
def test_select_instances_at_their_limits(ckv, many_heads, C_max):
    # the selection's instance follows the chunk capacity and whether the heads fit one wave: 4, 13 or
    # 16 keys a thread at 1024 threads, the keys in shared memory up to 32768 chunks and the general
    # kernel above; with more heads than SMs, 8 / 8 / 12 keys at 256 / 512 / 512 threads up to 6144
    # chunks.  Each limit and the next size,
    # bit-exact against the oracle on ragged sequences (one empty, one with a ragged last chunk
    # straddling the window), half of the heads with many tied scores
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    rng = np.random.default_rng(C_max + 7 * many_heads)
    Hkv, c, w = 4, 2, 17
    B = sms // Hkv + 2 if many_heads else 3
    lens = rng.integers(0, C_max * c + 1, size=B)
    lens[0], lens[1], lens[2] = C_max * c, 0, C_max * c - 1
    cu = [0] + list(itertools.accumulate(int(x) for x in lens))
    L_max = C_max * c * 3 // 10
    p, keep = ckv.make_params(cu_seqlens=cu, Hq=Hkv, Hkv=Hkv, d=64, w=w, c=c, L_max=L_max, dtype=torch.bfloat16)
    n_cap, c_max = ckv.chunkkv_out_capacity(p)
    assert c_max == C_max
    scores = rng.standard_normal((B, Hkv, C_max)).astype(np.float32)
    scores[:, ::2] = rng.integers(-3, 6, size=(B, (Hkv + 1) // 2, C_max)).astype(np.float32) * 0.125
    indices = torch.full((B, Hkv, n_cap), -1, dtype=torch.int32, device=DEV)
    counts = torch.zeros(B, Hkv, dtype=torch.int32, device=DEV)
    ckv.chunkkv_select(p, torch.from_numpy(scores).to(DEV), indices, counts)
    torch.cuda.synchronize()
    del keep
    indices, counts = indices.cpu().numpy(), counts.cpu().numpy()
    for b in sorted({0, 1, 2, B - 1, int(rng.integers(3, B))} if B > 3 else {0, 1, 2}):
        T = int(lens[b])
        C = -(-T // c)
        for h in range(Hkv):
            A = scores[b, h, :C].astype(np.float64)
            want = oracle.kept_indices(oracle.top_chunks(A, oracle.n_select(T, c, L_max)), T, c, w)
            n = int(counts[b, h])
            assert n == len(want), (b, h)
            assert np.array_equal(indices[b, h, :n], want), (b, h)


def test_window_queries_in_pinned_host_memory(ckv):
    # Q_w may be host memory the GPU addresses.  With w dividing 128 the scoring kernel reads device Q_w
    # through a tensor map; host Q_w goes through the packing kernel's plain loads instead (one launch
    # more).  Checked against the oracle like every other path.
    wl = configs.llama_model().with_params(seqlens=(3000, 1234), B=2, n_layers=4, n_reuse=2, L_max=600,
                                           name="host_q")
    qs, ks, vs, spans = gen.make_all_layers(wl, DEV)
    hq = [None if q is None else q.cpu().pin_memory() for q in qs]
    n0 = ckv.chunkkv_launch_count()
    run_and_check(ckv, wl, qs=hq, ks=ks, vs=vs, spans=spans)
    host_launches = ckv.chunkkv_launch_count() - n0
    n0 = ckv.chunkkv_launch_count()
    run_and_check(ckv, wl, qs=qs, ks=ks, vs=vs, spans=spans)
    assert host_launches == ckv.chunkkv_launch_count() - n0 + 1


def _rescale_inputs(T, Hq, Hkv, w, d, spike_every, spike_at, seed=5):
    """Window queries half along a per-head direction u and half against it (alternating window rows),
    low-magnitude keys, and every spike_every keys (from spike_at) a key of length 34 along u."""
    g = torch.Generator().manual_seed(seed)
    G = Hq // Hkv
    u = torch.randn(Hkv, d, generator=g, dtype=torch.float64)
    u /= u.norm(dim=1, keepdim=True)
    sign = torch.where(torch.arange(w) % 2 == 0, 1.0, -1.0).double()
    q = torch.randn(1, w, Hq, d, generator=g, dtype=torch.float64)
    q += 10.0 * sign[None, :, None, None] * u.repeat_interleave(G, 0)[None, None]
    k = 0.3 * torch.randn(T, Hkv, d, generator=g, dtype=torch.float64)
    pos = torch.arange(spike_at, T - w, spike_every)
    k[pos] = 34.0 * u[None]
    v = torch.randn(T, Hkv, d, generator=g, dtype=torch.float64)
    return q, k, v, pos


def test_rows_that_outgrow_their_first_tile_reference(ckv):
    # The scoring kernel takes a row's reference from the first key tile of a work item; when a later
    # tile outgrows it by 2^23 the row moves its reference and rescales the bins it already wrote.
    # Rows along u meet a key about 30 (natural-log units) above their first tile's maximum past the
    # first tile of every work item; rows against u do not, so each warp holds both kinds.
    wl = configs.llama_layer().with_params(needles=NeedleSpec(kind="none"), name="rescale")
    q, k, v, _ = _rescale_inputs(wl.T_total, wl.Hq, wl.Hkv, wl.w, wl.d, 240, 150)
    qs, ks, vs = [x.to(torch.bfloat16).to(DEV) for x in (q, k, v)]
    run_and_check(ckv, wl, qs=[qs], ks=[ks], vs=[vs])


def test_causal_window_through_the_head_kernel(ckv):
    # 5 ragged sequences (one empty, two shorter than the window) x 8 KV heads x 3 reuse groups = 120
    # heads take the fused head kernel; with the causal window, rows at negative positions see no key
    # and carry an empty (R, sum) pair into its log-sum-exp
    seqlens = (3000, 77, 5, 4096, 0)
    wl = configs.mistral_ragged().with_params(seqlens=seqlens, B=len(seqlens), n_layers=6, n_reuse=2, L_max=600,
                                              needles=NeedleSpec(kind="none"), name="causal_head")
    n0 = ckv.chunkkv_launch_count()
    run_and_check(ckv, wl, causal=True)
    assert ckv.chunkkv_launch_count() - n0 == 3                    # score, head_kernel, gather
