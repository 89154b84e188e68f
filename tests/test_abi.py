"""The C ABI on the host: the library loads, exports every declared symbol, and rejects bad
arguments with status codes before touching the GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest

import llama_decoder_block_fwd_gb300 as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(llama_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = L.lib()
    names = declared_functions()
    assert "llama_block_forward" in names and "llama_stack_decode_step" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for code in range(8):
        assert L.llama_status_string(code) != "unknown status"
    assert L.llama_status_string(99) == "unknown status"


def test_bounds_checking_build_flag_plumbing():
    """The -DLLAMA_DEBUG build: _build.build(debug=True) compiles every source with the flag into
    its own library; that library reports the bounds checks in llama_build_info() and the release
    library does not; every translation unit defines the reader of its bounds word, which
    llama_get_device_status collects; the bounds status code has its name.  (No kernel runs here.)"""
    import subprocess

    from llama_decoder_block_fwd_gb300 import _build
    path = _build.build(debug=True)
    assert path == _build.LIB_DEBUG and os.path.exists(path)
    log = open(os.path.join(_build.BUILD_DEBUG, "ptxas.log")).read()
    assert all(f"== {src}" in log for src in _build.SOURCES)
    dbg = ctypes.CDLL(path)
    dbg.llama_build_info.restype = ctypes.c_int
    assert dbg.llama_build_info() == L.BUILD_BOUNDS_CHECKS
    if not L.DEBUG_BUILD:
        assert L.llama_build_info() == 0                      # the release library has no checks
    dbg.llama_status_string.restype = ctypes.c_char_p
    assert b"bounds" in dbg.llama_status_string(7)
    assert L.STATUS_NAMES[7] == "LLAMA_ERR_BOUNDS"
    syms = subprocess.run(["nm", "-C", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    for src in _build.SOURCES:
        assert f"llama::bounds_read_clear_{src[:-3]}()" in syms, src
    for name in declared_functions():                       # the same C ABI in both builds
        assert hasattr(dbg, name), name


def _dims(**kw):
    base = dict(B=1, S=4, d_model=16, n_q=8, n_kv=2, head_dim=2, d_ff=48, theta_base=1e4, eps=1e-5)
    base.update(kw)
    return L.dims_of(**base)


def test_rejects_bad_arguments_without_launching():
    lib = L.lib()
    d = _dims()
    fake = 0x10000  # aligned, never dereferenced: validation fails before any launch
    # null pointers
    assert lib.llama_rmsnorm(ctypes.byref(d), L.F32, None, fake, fake, None) == 1
    # bad dtype
    assert lib.llama_rmsnorm(ctypes.byref(d), 7, fake, fake, fake, None) == 2
    # misaligned
    assert lib.llama_rmsnorm(ctypes.byref(d), L.F32, fake + 4, fake, fake, None) == 3
    # n_q not a multiple of n_kv
    bad = _dims(n_kv=3)
    assert lib.llama_rope(ctypes.byref(bad), L.F32, fake, fake, 0, None) == 1
    # odd head_dim
    assert lib.llama_rope(ctypes.byref(_dims(head_dim=3)), L.F32, fake, fake, 0, None) == 1
    # negative sizes
    assert lib.llama_rmsnorm(ctypes.byref(_dims(B=-1)), L.F32, fake, fake, fake, None) == 1
    # attention past the cache capacity
    assert lib.llama_gqa_attention(ctypes.byref(d), L.F32, fake, fake, fake, 3, 0, fake, None, 0, None) == 1
    # workspace missing / too small
    assert lib.llama_swiglu_ffn(ctypes.byref(d), L.F32, fake, fake, fake, fake, fake + 256, None, 0, None) == 4
    need = L.llama_workspace_bytes(L.OP_SWIGLU_FFN, d, L.F32)
    assert need >= 4 * 48 * 4
    assert lib.llama_swiglu_ffn(ctypes.byref(d), L.F32, fake, fake, fake, fake, fake + 256, fake, need - 1, None) == 4
    # aliasing input and output
    assert lib.llama_swiglu_ffn(ctypes.byref(d), L.F32, fake, fake, fake, fake, fake, fake, need, None) == 1
    # decode needs S == 1
    w = (L.BlockWeights * 1)(L.BlockWeights(*[fake] * 9))
    assert lib.llama_stack_decode_step(ctypes.byref(d), L.F32, 1, w, fake, fake, 10, fake, fake, fake, 8, 4, fake,
                                       fake, 1 << 20, None) == 1
    # block with pos0 > 0 but no cache
    bw = L.BlockWeights(*[fake] * 9)
    assert lib.llama_block_forward(ctypes.byref(d), L.F32, ctypes.byref(bw), fake, fake + 256, 2, None, None, 0,
                                   fake, 1 << 20, None) == 1
    # one cache only
    assert lib.llama_block_forward(ctypes.byref(d), L.F32, ctypes.byref(bw), fake, fake + 256, 0, fake, None, 8,
                                   fake, 1 << 20, None) == 1


def test_empty_inputs_are_no_ops():
    lib = L.lib()
    d = _dims(B=0)
    assert lib.llama_rmsnorm(ctypes.byref(d), L.F32, None, None, None, None) == 0
    assert lib.llama_rope(ctypes.byref(_dims(S=0)), L.BF16, None, None, 0, None) == 0


def test_workspace_sizes_grow_with_shape():
    small = L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, _dims(), L.BF16)
    big = L.llama_workspace_bytes(L.OP_BLOCK_FORWARD, _dims(S=400), L.BF16)
    assert 0 < small < big
    assert L.llama_workspace_bytes(L.OP_STACK_DECODE_STEP, _dims(B=64, S=1), L.BF16) > 0
    assert L.llama_workspace_bytes(L.OP_RMSNORM, _dims(), L.BF16) == 0


def test_sample_and_embed_reject_bad_arguments():
    lib = L.lib()
    fake = 0x10000
    nan = float("nan")
    # B < 0, vocab < 1, ld < vocab, NaN temperature / top_p, NULL pointers
    assert lib.llama_sample(fake, -1, 10, 10, 1.0, 0, 1.0, fake, fake, None) == 1
    assert lib.llama_sample(fake, 2, 0, 10, 1.0, 0, 1.0, fake, fake, None) == 1
    assert lib.llama_sample(fake, 2, 10, 5, 1.0, 0, 1.0, fake, fake, None) == 1
    assert lib.llama_sample(fake, 2, 10, 10, nan, 0, 1.0, fake, fake, None) == 1
    assert lib.llama_sample(fake, 2, 10, 10, 1.0, 0, nan, fake, fake, None) == 1
    assert lib.llama_sample(None, 2, 10, 10, 1.0, 0, 1.0, fake, fake, None) == 1
    assert lib.llama_sample(fake + 2, 2, 10, 10, 1.0, 0, 1.0, fake, fake, None) == 3
    assert lib.llama_sample(None, 0, 10, 10, 1.0, 0, 1.0, None, None, None) == 0   # nothing to do
    assert lib.llama_embed(7, fake, 10, 16, fake, 4, fake, None) == 2
    assert lib.llama_embed(L.BF16, fake, 0, 16, fake, 4, fake, None) == 1
    assert lib.llama_embed(L.BF16, fake, 10, 0, fake, 4, fake, None) == 1
    assert lib.llama_embed(L.BF16, None, 10, 16, fake, 4, fake, None) == 1
    assert lib.llama_embed(L.BF16, None, 10, 16, None, 0, None, None) == 0


def test_kv8_calls_reject_bad_arguments():
    lib = L.lib()
    fake = 0x10000
    d1 = _dims(S=1, n_q=32, n_kv=8, head_dim=128, d_model=4096)
    # llama_kv_quantize: head_dim not a multiple of 8, NULL scale, misaligned codes
    assert lib.llama_kv_quantize(fake, 4, 8, 12, fake, fake, None) == 1
    assert lib.llama_kv_quantize(fake, 4, 8, 128, None, fake, None) == 1
    assert lib.llama_kv_quantize(fake, 4, 8, 128, fake, fake + 4, None) == 3
    assert lib.llama_kv_quantize(None, 0, 8, 128, None, None, None) == 0
    # attention over codes: S != 1, pos0 beyond capacity, NULL scales, missing workspace
    d2 = _dims(S=2, n_q=32, n_kv=8, head_dim=128, d_model=4096)
    assert lib.llama_gqa_attention_decode_kv8(ctypes.byref(d2), fake, fake, fake, fake, fake, 100, 10, fake, fake, 1 << 20, None) == 1
    assert lib.llama_gqa_attention_decode_kv8(ctypes.byref(d1), fake, fake, fake, fake, fake, 100, 100, fake, fake, 1 << 20, None) == 1
    assert lib.llama_gqa_attention_decode_kv8(ctypes.byref(d1), fake, fake, fake, None, fake, 100, 10, fake, fake, 1 << 20, None) == 1
    # head_dim 64 is not supported on this path
    d3 = _dims(S=1, n_q=8, n_kv=2, head_dim=64, d_model=512)
    assert lib.llama_gqa_attention_decode_kv8(ctypes.byref(d3), fake, fake, fake, fake, fake, 100, 10, fake, fake, 1 << 20, None) == 2
    # the stack call needs kv_scales
    w = (L.BlockWeights * 1)(L.BlockWeights(*([fake] * 9)))
    dd = _dims(B=4, S=1, n_q=32, n_kv=8, head_dim=128, d_model=4096, d_ff=14336)
    assert lib.llama_stack_decode_step_kv8(ctypes.byref(dd), 1, w, fake, fake, 128, fake, fake, fake, None, 100, 10,
                                           fake, fake, 1 << 30, None) == 1


def test_host_tensors_are_refused_before_the_library_is_called():
    """Every pointer of the ABI is device memory; the binding refuses a host tensor up front."""
    torch = pytest.importorskip("torch")
    d = _dims()
    x = torch.zeros(4, 16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.llama_rmsnorm(d, L.F32, x, torch.ones(16), torch.empty_like(x), stream=0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.llama_sample(torch.zeros(2, 10), 1.0, 0, 1.0, torch.zeros(2), torch.zeros(2, dtype=torch.int32), stream=0)


def test_block_weights_keep_their_tensors_alive():
    """The weight struct holds raw addresses; it also keeps references to the tensors it was built
    from, so dropping the caller's dict does not free memory the library still reads."""
    import gc
    import weakref

    class FakeDeviceTensor:   # what _p needs: is_cuda and data_ptr
        is_cuda = True

        def __init__(self, addr):
            self.addr = addr

        def data_ptr(self):
            return self.addr

    w = {n: FakeDeviceTensor(0x1000 * (i + 1)) for i, n in enumerate(L._WEIGHT_FIELDS)}
    refs = [weakref.ref(t) for t in w.values()]
    bw = L.block_weights(w)
    del w
    gc.collect()
    assert all(r() is not None for r in refs)
    assert [getattr(bw, n) for n in L._WEIGHT_FIELDS] == [0x1000 * (i + 1) for i in range(len(L._WEIGHT_FIELDS))]
    del bw
    gc.collect()
    assert all(r() is None for r in refs)


def _noalloc_scratch_bytes(B, n_kv, r):
    """The allocation-free decode attention's size rule as its header states it: B*n_kv + 256
    slots of r rows of 130 floats, as two arrays each rounded up to 256 bytes."""
    r256 = lambda b: (b + 255) // 256 * 256
    slots = B * n_kv + 256
    return r256(slots * r * 512) + r256(slots * r * 8)


@pytest.mark.parametrize("n_q,n_kv", [(32, 8), (64, 4)])   # r = 4 and r = 16
def test_noalloc_size_rule_at_its_boundary(n_q, n_kv):
    """Just under the 12 MiB rule the call gets past the size check (and, with no GPU visible in
    the child process, stops at its first CUDA call: LLAMA_ERR_CUDA); just over it returns
    LLAMA_ERR_WORKSPACE.  The number of keys does not enter the rule."""
    import subprocess
    import sys
    r = n_q // n_kv
    B = 1
    while _noalloc_scratch_bytes(B + 1, n_kv, r) <= 12 << 20:
        B += 1
    code = f"""
import ctypes, sys
sys.path.insert(0, {ROOT!r})
import llama_decoder_block_fwd_gb300 as L
lib = L.lib()
fake = 0x10000
out = []
for B in ({B}, {B + 1}):
    for keys in (1, 100000):
        d = L.dims_of(B, 1, {n_q} * 128, {n_q}, {n_kv}, 128, 1, 5e5, 1e-5)
        out.append(lib.llama_gqa_attention_decode_noalloc(ctypes.byref(d), L.BF16, fake, fake, fake, keys, keys - 1,
                                                          fake, None))
print(out)
"""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    rcs = eval(res.stdout.strip().splitlines()[-1])
    assert rcs[:2] == [5, 5], rcs      # under: past the size check, no device to reach
    assert rcs[2:] == [4, 4], rcs      # over: LLAMA_ERR_WORKSPACE
    if (n_q, n_kv) == (32, 8):
        assert B == 724                # the largest batch the header names for 32/8 heads
