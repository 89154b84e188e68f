"""Python binding of the C ABI in include/llama_block.h.

Argument marshalling only: every step of the block runs in the CUDA kernels of
libllama_block.so.  torch is used for device memory and streams; tensors are
passed as raw device pointers.  If the library has not been built the first
call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Sequence

__all__ = [
    "F32", "BF16", "X_F32", "Y_F32", "LlamaError", "Dims", "BlockWeights", "lib", "dims_of",
    "llama_rmsnorm", "llama_rope", "llama_gqa_attention", "llama_gqa_attention_decode_noalloc", "llama_swiglu_ffn",
    "llama_block_forward", "llama_stack_decode_step", "llama_workspace_bytes",
    "llama_sample", "llama_embed", "llama_kv_quantize", "llama_gqa_attention_decode_kv8",
    "llama_stack_decode_step_kv8", "llama_stack_decode_step_paged", "llama_gqa_attention_decode_paged",
    "llama_get_device_status", "llama_status_string", "llama_profile_enable", "llama_profile_read",
    "llama_selftest_bounded_wait", "llama_selftest_bounds", "llama_build_info", "BUILD_BOUNDS_CHECKS", "DEBUG_BUILD",
    "OP_RMSNORM", "OP_ROPE", "OP_GQA_ATTENTION", "OP_SWIGLU_FFN", "OP_BLOCK_FORWARD",
    "OP_STACK_DECODE_STEP",
]

F32, BF16 = 0, 1
X_F32, Y_F32 = 0x100, 0x200   # residual-stream flags for llama_block_forward's dtype (x fp32, y fp32)
(OP_RMSNORM, OP_ROPE, OP_GQA_ATTENTION, OP_SWIGLU_FFN, OP_BLOCK_FORWARD,
 OP_STACK_DECODE_STEP) = range(6)
STATUS_NAMES = {0: "LLAMA_OK", 1: "LLAMA_ERR_INVALID_ARG", 2: "LLAMA_ERR_UNSUPPORTED",
                3: "LLAMA_ERR_ALIGNMENT", 4: "LLAMA_ERR_WORKSPACE", 5: "LLAMA_ERR_CUDA",
                6: "LLAMA_ERR_TIMEOUT", 7: "LLAMA_ERR_BOUNDS"}

_DIR = os.path.dirname(os.path.abspath(__file__))
# LLAMA_BLOCK_DEBUG=1 selects the bounds-checking build (built by _build.build(debug=True))
DEBUG_BUILD = os.environ.get("LLAMA_BLOCK_DEBUG", "0") not in ("", "0")
LIB_PATH = os.path.join(_DIR, "libllama_block_debug.so" if DEBUG_BUILD else "libllama_block.so")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("S", ctypes.c_int64), ("d_model", ctypes.c_int64),
                ("n_q", ctypes.c_int64), ("n_kv", ctypes.c_int64), ("head_dim", ctypes.c_int64),
                ("d_ff", ctypes.c_int64), ("theta_base", ctypes.c_double), ("eps", ctypes.c_double)]


_WEIGHT_FIELDS = ["attn_norm_g", "wq", "wk", "wv", "wo", "ffn_norm_g", "w_gate", "w_up", "w_down"]


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class LlamaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was not built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            pd = ctypes.POINTER(Dims)
            sig = {
                "llama_rmsnorm": [pd, i32, vp, vp, vp, vp],
                "llama_rope": [pd, i32, vp, vp, i64, vp],
                "llama_gqa_attention": [pd, i32, vp, vp, vp, i64, i64, vp, vp, sz, vp],
                "llama_swiglu_ffn": [pd, i32, vp, vp, vp, vp, vp, vp, sz, vp],
                "llama_block_forward": [pd, i32, ctypes.POINTER(BlockWeights), vp, vp, i64, vp, vp, i64,
                                        vp, sz, vp],
                "llama_stack_decode_step": [pd, i32, i32, ctypes.POINTER(BlockWeights), vp, vp, i64, vp,
                                            vp, vp, i64, i64, vp, vp, sz, vp],
                "llama_get_device_status": [ctypes.POINTER(ctypes.c_int), vp],
                "llama_selftest_bounded_wait": [vp],
                "llama_selftest_bounds": [vp, vp],
                "llama_gqa_attention_decode_noalloc": [pd, i32, vp, vp, vp, i64, i64, vp, vp],
                "llama_sample": [vp, i64, i64, i64, ctypes.c_float, i64, ctypes.c_float, vp, vp, vp],
                "llama_embed": [i32, vp, i64, i64, vp, i64, vp, vp],
                "llama_kv_quantize": [vp, i64, i64, i64, vp, vp, vp],
                "llama_gqa_attention_decode_kv8": [pd, vp, vp, vp, vp, vp, i64, i64, vp, vp, sz, vp],
                "llama_stack_decode_step_kv8": [pd, i32, ctypes.POINTER(BlockWeights), vp, vp, i64, vp, vp, vp, vp,
                                                i64, i64, vp, vp, sz, vp],
                "llama_stack_decode_step_paged": [pd, i32, ctypes.POINTER(BlockWeights), vp, vp, i64, vp, vp, vp,
                                                  i64, vp, i64, vp, i64, vp, vp, sz, vp],
                "llama_gqa_attention_decode_paged": [pd, vp, vp, vp, i64, vp, i64, vp, i64, vp, vp, sz, vp],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.llama_workspace_bytes.argtypes = [i32, pd, i32, i32, i64, i64]
            L.llama_workspace_bytes.restype = sz
            L.llama_profile_enable.argtypes = [i32]
            L.llama_profile_enable.restype = ctypes.c_int
            L.llama_profile_read.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
            L.llama_profile_read.restype = ctypes.c_int
            L.llama_build_info.argtypes = []
            L.llama_build_info.restype = ctypes.c_int
            L.llama_status_string.argtypes = [i32]
            L.llama_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def dims_of(B, S, d_model, n_q, n_kv, head_dim, d_ff, theta_base, eps) -> Dims:
    return Dims(int(B), int(S), int(d_model), int(n_q), int(n_kv), int(head_dim), int(d_ff),
                float(theta_base), float(eps))


def _d(dims) -> Dims:
    if isinstance(dims, Dims):
        return dims
    if isinstance(dims, Sequence):
        return dims_of(*dims)
    return dims_of(dims.B, dims.S, dims.d_model, dims.n_q, dims.n_kv, dims.head_dim, dims.d_ff,
                   dims.theta_base, dims.eps)


def _p(t) -> int | None:
    """The device address of a tensor (an int passes through as an address).  Every pointer of the
    C ABI is device memory: a tensor that lives on the host is refused here, not handed to a kernel."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"expected a CUDA tensor, got one on {getattr(t, 'device', type(t).__name__)}")
    return t.data_ptr()


def _s(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise LlamaError(rc, where)


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def block_weights(w) -> BlockWeights:
    """BlockWeights from a mapping (or object) holding the nine device tensors.  The struct keeps
    references to the tensors, so their memory stays allocated while the struct is alive (the
    library reads it through the raw pointers)."""
    get = (lambda n: w[n]) if isinstance(w, dict) else (lambda n: getattr(w, n))
    tensors = [get(n) for n in _WEIGHT_FIELDS]
    bw = BlockWeights(*[_p(t) for t in tensors])
    bw._tensors = tensors
    return bw


def llama_rmsnorm(dims, dtype, x, g, y, stream=None):
    _check(lib().llama_rmsnorm(ctypes.byref(_d(dims)), dtype, _p(x), _p(g), _p(y), _s(stream)), "llama_rmsnorm")


def llama_rope(dims, dtype, q, k, pos0=0, stream=None):
    _check(lib().llama_rope(ctypes.byref(_d(dims)), dtype, _p(q), _p(k), int(pos0), _s(stream)), "llama_rope")


def llama_gqa_attention(dims, dtype, q, k, v, kv_capacity, pos0, o, ws=None, stream=None):
    _check(lib().llama_gqa_attention(ctypes.byref(_d(dims)), dtype, _p(q), _p(k), _p(v), int(kv_capacity),
                                     int(pos0), _p(o), _p(ws), _nbytes(ws), _s(stream)), "llama_gqa_attention")


def llama_gqa_attention_decode_noalloc(dims, dtype, q, k, v, kv_capacity, pos0, o, stream=None):
    """One-token attention with the library's own fixed scratch (no workspace argument)."""
    _check(lib().llama_gqa_attention_decode_noalloc(ctypes.byref(_d(dims)), dtype, _p(q), _p(k), _p(v),
                                                    int(kv_capacity), int(pos0), _p(o), _s(stream)),
           "llama_gqa_attention_decode_noalloc")


def llama_swiglu_ffn(dims, dtype, x, w_gate, w_up, w_down, y, ws, stream=None):
    _check(lib().llama_swiglu_ffn(ctypes.byref(_d(dims)), dtype, _p(x), _p(w_gate), _p(w_up), _p(w_down),
                                  _p(y), _p(ws), _nbytes(ws), _s(stream)), "llama_swiglu_ffn")


def llama_block_forward(dims, dtype, weights, x, y, pos0=0, k_cache=None, v_cache=None, cache_capacity=0,
                        ws=None, stream=None):
    w = weights if isinstance(weights, BlockWeights) else block_weights(weights)
    _check(lib().llama_block_forward(ctypes.byref(_d(dims)), dtype, ctypes.byref(w), _p(x), _p(y), int(pos0),
                                     _p(k_cache), _p(v_cache), int(cache_capacity), _p(ws), _nbytes(ws),
                                     _s(stream)), "llama_block_forward")


def llama_stack_decode_step(dims, dtype, layers, final_g, w_lm, vocab, x_emb, k_cache, v_cache, cache_capacity,
                            t_cache, logits, ws, stream=None):
    n = len(layers)
    arr = (BlockWeights * n)(*[lw if isinstance(lw, BlockWeights) else block_weights(lw) for lw in layers])
    _check(lib().llama_stack_decode_step(ctypes.byref(_d(dims)), dtype, n, arr, _p(final_g), _p(w_lm), int(vocab),
                                         _p(x_emb), _p(k_cache), _p(v_cache), int(cache_capacity), int(t_cache),
                                         _p(logits), _p(ws), _nbytes(ws), _s(stream)), "llama_stack_decode_step")


def llama_sample(logits, temperature, top_k, top_p, u, tokens, vocab=None, stream=None):
    """tokens[b] <- the token chosen from logits[b, :vocab] (fp32 [B, ld]) with the uniform u[b]."""
    B = 0 if logits is None else int(logits.shape[0])
    ld = 0 if logits is None else int(logits.stride(0))
    V = int(logits.shape[1]) if vocab is None else int(vocab)
    _check(lib().llama_sample(_p(logits), B, V, ld, float(temperature), int(top_k), float(top_p), _p(u), _p(tokens),
                              _s(stream)), "llama_sample")


def llama_embed(dtype, table, tokens, x, stream=None):
    """x[i] <- table[tokens[i]] (table [vocab, d_model], tokens int32 [n], x [n, d_model])."""
    _check(lib().llama_embed(dtype, _p(table), int(table.shape[0]), int(table.shape[1]), _p(tokens),
                             int(tokens.numel()), _p(x), _s(stream)), "llama_embed")


def llama_kv_quantize(x, scale, codes, stream=None):
    """codes <- E4M3(x / scale[head]) for x bf16 [..., n_kv, head_dim], scale fp32 [n_kv]."""
    n_kv, hd = int(x.shape[-2]), int(x.shape[-1])
    _check(lib().llama_kv_quantize(_p(x), int(x.numel() // (n_kv * hd)), n_kv, hd, _p(scale), _p(codes), _s(stream)),
           "llama_kv_quantize")


def llama_gqa_attention_decode_kv8(dims, q, k, v, k_scale, v_scale, kv_capacity, pos0, o, ws, stream=None):
    _check(lib().llama_gqa_attention_decode_kv8(ctypes.byref(_d(dims)), _p(q), _p(k), _p(v), _p(k_scale),
                                                _p(v_scale), int(kv_capacity), int(pos0), _p(o), _p(ws), _nbytes(ws),
                                                _s(stream)), "llama_gqa_attention_decode_kv8")


def llama_stack_decode_step_kv8(dims, layers, final_g, w_lm, vocab, x_emb, k_cache, v_cache, kv_scales,
                                cache_capacity, t_cache, logits, ws, stream=None):
    n = len(layers)
    arr = (BlockWeights * n)(*[lw if isinstance(lw, BlockWeights) else block_weights(lw) for lw in layers])
    _check(lib().llama_stack_decode_step_kv8(ctypes.byref(_d(dims)), n, arr, _p(final_g), _p(w_lm), int(vocab),
                                             _p(x_emb), _p(k_cache), _p(v_cache), _p(kv_scales), int(cache_capacity),
                                             int(t_cache), _p(logits), _p(ws), _nbytes(ws), _s(stream)),
           "llama_stack_decode_step_kv8")


def llama_stack_decode_step_paged(dims, layers, final_g, w_lm, vocab, x_emb, k_pool, v_pool, block_table, seq_pos,
                                  max_pos, logits, ws, stream=None):
    """k_pool / v_pool [n_layers, n_pages, 128, n_kv, hd] bf16; block_table int32 [B, max_pages]."""
    n = len(layers)
    arr = (BlockWeights * n)(*[lw if isinstance(lw, BlockWeights) else block_weights(lw) for lw in layers])
    _check(lib().llama_stack_decode_step_paged(ctypes.byref(_d(dims)), n, arr, _p(final_g), _p(w_lm), int(vocab),
                                               _p(x_emb), _p(k_pool), _p(v_pool), int(k_pool.shape[1]),
                                               _p(block_table), int(block_table.shape[1]), _p(seq_pos), int(max_pos),
                                               _p(logits), _p(ws), _nbytes(ws), _s(stream)),
           "llama_stack_decode_step_paged")


def llama_gqa_attention_decode_paged(dims, q, k_pool, v_pool, block_table, seq_pos, max_pos, o, ws, stream=None):
    """k_pool / v_pool [n_pages, 128, n_kv, hd] bf16 (one layer); block_table int32 [B, max_pages]."""
    _check(lib().llama_gqa_attention_decode_paged(ctypes.byref(_d(dims)), _p(q), _p(k_pool), _p(v_pool),
                                                  int(k_pool.shape[0]), _p(block_table), int(block_table.shape[1]),
                                                  _p(seq_pos), int(max_pos), _p(o), _p(ws), _nbytes(ws), _s(stream)),
           "llama_gqa_attention_decode_paged")


def llama_workspace_bytes(op, dims, dtype, n_layers=0, vocab=0, kv_capacity=0) -> int:
    return int(lib().llama_workspace_bytes(int(op), ctypes.byref(_d(dims)), dtype, int(n_layers), int(vocab),
                                           int(kv_capacity)))


def llama_get_device_status(stream=None) -> int:
    out = ctypes.c_int(-1)
    _check(lib().llama_get_device_status(ctypes.byref(out), _s(stream)), "llama_get_device_status")
    return out.value


def llama_selftest_bounded_wait(stream=None) -> None:
    """Launch the kernel whose bounded waits run out on purpose (the device status word then holds
    LLAMA_ERR_TIMEOUT; read it with llama_get_device_status)."""
    _check(lib().llama_selftest_bounded_wait(_s(stream)), "llama_selftest_bounded_wait")


def llama_selftest_bounds(scratch, stream=None) -> None:
    """Store through the checked path to element 40 of `scratch` (64 fp32) declared 32 long: a
    bounds-checking build skips it and latches LLAMA_ERR_BOUNDS, a release build performs it."""
    _check(lib().llama_selftest_bounds(_p(scratch), _s(stream)), "llama_selftest_bounds")


def llama_build_info() -> int:
    """Bit 1 (LLAMA_BUILD_BOUNDS_CHECKS): the loaded library checks bounds (-DLLAMA_DEBUG)."""
    return int(lib().llama_build_info())


BUILD_BOUNDS_CHECKS = 1


def llama_profile_enable(on: bool = True) -> None:
    _check(lib().llama_profile_enable(1 if on else 0), "llama_profile_enable")


def llama_profile_read(max_kinds: int = 32) -> dict:
    """{kernel role: (launches, total_ms)} for the launches recorded since the last read."""
    names = (ctypes.c_char_p * max_kinds)()
    launches = (ctypes.c_int * max_kinds)()
    ms = (ctypes.c_double * max_kinds)()
    n = ctypes.c_int(0)
    _check(lib().llama_profile_read(max_kinds, names, launches, ms, ctypes.byref(n)), "llama_profile_read")
    return {names[i].decode(): (launches[i], ms[i]) for i in range(n.value)}


def llama_status_string(status: int) -> str:
    return lib().llama_status_string(int(status)).decode()
