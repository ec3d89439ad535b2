"""The five synthetic workloads, sized like the models the ChunkKV evaluation uses.

The ChunkKV notes evaluate on LLaMA-3-8B, Mistral-7B and Qwen2-7B with
LongBench / NIAH style long prompts (§5.1 "实验设置"), chunk size c = 10 by
default and ablations over c in {3, 5, 10, 20, 30}, KV budgets given as a
ratio of the prompt (10 %, 20 %) or as a fixed size (128, 256, 512).  No
dataset content is used: every tensor is drawn by synthetic.generator, and
planted needle spans stand in for the retrieval targets.
"""
from __future__ import annotations

from .generator import HostStream, NeedleSpec, Workload, stream_key


def tiny() -> Workload:
    """One layer, GQA group 2, fp32, one planted chunk (the oracle runs it in ms)."""
    return Workload(name="tiny_f32_T512", B=1, Hq=4, Hkv=2, d=64, seqlens=(512,), dtype="f32",
                    w=8, c=10, L_max=128, n_layers=1, n_reuse=1, seed=1001,
                    needles=NeedleSpec(kind="chunk", count=1))


def llama_layer() -> Workload:
    """LLaMA-3-8B-shaped single prefill layer, T = 8192, 10 % budget."""
    return Workload(name="llama3_8b_layer_T8192", B=1, Hq=32, Hkv=8, d=128, seqlens=(8192,),
                    dtype="bf16", w=32, c=10, L_max=819, n_layers=1, n_reuse=1, seed=1002,
                    channel_scale=True, needles=NeedleSpec(kind="spans", count=20))


def llama_model() -> Workload:
    """LLaMA-3-8B-shaped 32-layer model, T = 32768, 20 % budget, N_reuse = 2."""
    T = 32768
    return Workload(name="llama3_8b_32L_T32768", B=1, Hq=32, Hkv=8, d=128, seqlens=(T,),
                    dtype="bf16", w=32, c=10, L_max=(T * 20) // 100, n_layers=32, n_reuse=2,
                    seed=1003, channel_scale=True,
                    needles=NeedleSpec(kind="spans", count=20, keep_across_layers=16))


def mistral_ragged(c: int = 10, L_max: int = 256) -> Workload:
    """Mistral-7B-shaped batch of 16 ragged prompts, T_b uniform in [4096, 16384]."""
    rs = HostStream(stream_key(1004, 555))
    seqlens = tuple(rs.randint(4096, 16384) for _ in range(16))
    return Workload(name=f"mistral_7b_32L_B16_ragged_c{c}_L{L_max}", B=16, Hq=32, Hkv=8, d=128,
                    seqlens=seqlens, dtype="bf16", w=32, c=c, L_max=L_max, n_layers=32,
                    n_reuse=2, seed=1004, channel_scale=False,
                    needles=NeedleSpec(kind="spans", count=10))


MISTRAL_SWEEP = [(c, L) for c in (3, 5, 10, 20, 30) for L in (128, 256, 512)]


def qwen_128k() -> Workload:
    """Qwen2-7B-shaped 28-layer model, T = 131072, GQA group 7, 10 % budget."""
    T = 131072
    return Workload(name="qwen2_7b_28L_T131072", B=1, Hq=28, Hkv=4, d=128, seqlens=(T,),
                    dtype="bf16", w=64, c=10, L_max=(T * 10) // 100, n_layers=28, n_reuse=2,
                    seed=1005, channel_scale=True, needles=NeedleSpec(kind="spans", count=50))


ALL = {
    "tiny": tiny,
    "llama_layer": llama_layer,
    "llama_model": llama_model,
    "mistral_ragged": mistral_ragged,
    "qwen_128k": qwen_128k,
}
