"""The algorithmic work the bench divides by (the roofline's numerators), against figures worked
out by hand from the shapes: the seven projections of an 8B block hold 218,103,808 weights (the
size pin of "LLaMA-3 8B ...", section 六), causal attention touches S(S+1)/2 query-key pairs per
head, and a decode step reads every cached position of every layer once."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import configs as C  # noqa: E402


def test_prefill_flops_8b_block():
    f = bench.prefill_flops(C.LLAMA3_8B_PREFILL)
    assert f["gemm_tc_qkv"] + f["gemm_tc_resid"] + f["gemm_tc_swiglu"] == 2 * 8192 * 218_103_808
    assert f["attn"] == 4 * 32 * 128 * 8192 * 8193 // 2 == 549_822_922_752
    assert sum(f.values()) == 4_123_235_713_024


def test_prefill_flops_mha_block():
    f = bench.prefill_flops(C.LLAMA_7B_MHA_PREFILL)
    assert sum(v for k, v in f.items() if k != "attn") == 2 * 4 * 2048 * (4 * 4096 * 4096 + 3 * 4096 * 11008)
    assert f["attn"] == 4 * 32 * 128 * 4 * 2048 * 2049 // 2
    assert sum(f.values()) == 3_453_220_814_848


def test_decode_bytes_32_layer_step():
    b = bench.decode_bytes(C.LLAMA3_8B_DECODE)
    assert b["kv_read"] == 32 * 64 * 8193 * 8 * 128 * 2 * 2          # K and V of 8193 positions, bf16
    assert b["weights"] == 32 * 436_224_000                          # 218,112,000 parameters a layer, bf16
    assert b["lm_head"] == 128256 * 4096 * 2 + 4096 * 2
    assert sum(b.values()) == 83_779_461_120
    b8 = bench.decode_bytes(C.LLAMA3_8B_DECODE, kv_elem_bytes=1)    # E4M3 codes: half the cache bytes
    assert b8["kv_read"] * 2 == b["kv_read"]
