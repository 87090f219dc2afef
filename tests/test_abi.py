"""The C ABI without a GPU: the library loads, exports every declared symbol, and its
host-side checks reject bad arguments before anything is launched."""
import ctypes
import os
import re

import pytest

from block_wise_diffusion_denoise_b300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^TT_API\s+[\w\s\*]*?\b(tt_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    return N.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert len(declared) >= 10
    assert set(declared) == set(N.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code in range(7):
        assert lib.tt_status_string(code)
    assert lib.tt_status_string(99) == b"unknown status"
    assert lib.tt_version() >= 10000


def test_workspace_sizes(lib):
    n = ctypes.c_size_t(0)
    assert lib.tt_unmask_workspace_size(32, 16, 131072, N.TT_BF16, ctypes.byref(n)) == N.TT_OK
    # 8 vocabulary chunks of 16384 bf16 per row, 16-byte partials, plus the ticket words
    assert n.value >= 32 * 16 * 8 * 16 + 32 * 4
    assert lib.tt_unmask_workspace_size(-1, 16, 10, N.TT_BF16, ctypes.byref(n)) == N.TT_ERR_INVALID_ARG
    assert lib.tt_unmask_workspace_size(1, 2000, 10, N.TT_BF16, ctypes.byref(n)) == N.TT_ERR_UNSUPPORTED
    assert lib.tt_denoise_attn_workspace_size(4, 16, 32, 2, 128, N.TT_BF16, ctypes.byref(n)) == N.TT_OK
    assert lib.tt_denoise_attn_workspace_size(4, 16, 30, 4, 128, N.TT_BF16, ctypes.byref(n)) == N.TT_ERR_INVALID_ARG
    assert lib.tt_denoise_attn_workspace_size(4, 16, 32, 2, 96, N.TT_BF16, ctypes.byref(n)) == N.TT_ERR_UNSUPPORTED
    assert lib.tt_denoise_attn_workspace_size(4, 16, 32, 2, 128, 7, ctypes.byref(n)) == N.TT_ERR_INVALID_ARG
    assert lib.tt_denoise_attn_workspace_size(4, 16, 32, 2, 128, N.TT_BF16, None) == N.TT_ERR_INVALID_ARG
    # one position, 16 query heads per KV head: the decode kernel's split partials
    # (O^T of 16 heads x 128 d, then 16 maxima and 16 sums) for every CTA and segment
    assert lib.tt_denoise_attn_workspace_size(4, 1, 32, 2, 128, N.TT_BF16, ctypes.byref(n)) == N.TT_OK
    assert n.value >= (296 + 8) * (16 * 128 + 32) * 4
    # one position with another head ratio, or fp32: no tensor-core kernel, no workspace
    assert lib.tt_denoise_attn_workspace_size(4, 1, 16, 2, 128, N.TT_BF16, ctypes.byref(n)) == N.TT_OK
    assert n.value == 0
    assert lib.tt_denoise_attn_workspace_size(4, 1, 32, 2, 128, N.TT_FP32, ctypes.byref(n)) == N.TT_OK
    assert n.value == 0
    t = ctypes.c_size_t(0)
    a = ctypes.c_size_t(0)
    u = ctypes.c_size_t(0)
    assert lib.tt_block_step_workspace_size(8, 16, 32, 2, 128, 4096, N.TT_BF16, ctypes.byref(t)) == N.TT_OK
    lib.tt_denoise_attn_workspace_size(8, 16, 32, 2, 128, N.TT_BF16, ctypes.byref(a))
    lib.tt_unmask_workspace_size(8, 16, 4096, N.TT_BF16, ctypes.byref(u))
    assert t.value >= a.value + u.value


def _cache(**kw):
    c = N.tt_kv_cache()
    c.k_pool, c.v_pool, c.page_table, c.ctx_len = 0x1000, 0x2000, 0x3000, 0x4000
    c.num_pages, c.max_pages_per_seq, c.page_size, c.n_kv_heads, c.head_dim, c.dtype = 8, 4, 64, 2, 128, N.TT_BF16
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("entry", ["tt_denoise_attn", "tt_context_block_attn"])
def test_attention_rejects_bad_arguments_on_the_host(lib, entry):
    def call(cache, q=0x10000, B=1, S=16, Hq=32, scale=0.1, max_ctas=0):
        return getattr(lib, entry)(ctypes.byref(cache) if cache is not None else None, q, 0x20000, 0x30000,
                                   0x40000, None, B, S, Hq, scale, max_ctas, None, 0, None, None)
    assert call(None) == N.TT_ERR_INVALID_ARG
    assert call(_cache(page_table=0)) == N.TT_ERR_INVALID_ARG
    assert call(_cache(ctx_len=0)) == N.TT_ERR_INVALID_ARG
    assert call(_cache(page_size=0)) == N.TT_ERR_INVALID_ARG
    assert call(_cache(dtype=5)) == N.TT_ERR_INVALID_ARG
    assert call(_cache(head_dim=80)) == N.TT_ERR_UNSUPPORTED
    assert call(_cache(max_pages_per_seq=(1 << 24) + 1)) == N.TT_ERR_UNSUPPORTED   # > 2^30 tokens
    assert call(_cache(k_pool=0x1008)) == N.TT_ERR_UNSUPPORTED          # pool not 16-byte aligned
    assert call(_cache(), Hq=31) == N.TT_ERR_INVALID_ARG                # Hq not a multiple of Hkv
    assert call(_cache(), S=0) == N.TT_ERR_INVALID_ARG
    assert call(_cache(), B=-1) == N.TT_ERR_INVALID_ARG
    assert call(_cache(), q=0) == N.TT_ERR_INVALID_ARG
    assert call(_cache(), q=0x10004) == N.TT_ERR_UNSUPPORTED            # q not 16-byte aligned
    assert call(_cache(), scale=float("nan")) == N.TT_ERR_INVALID_ARG
    assert call(_cache(), max_ctas=-1) == N.TT_ERR_INVALID_ARG
    assert call(_cache(), B=0) == N.TT_OK                               # nothing to do, nothing launched


def test_unmask_rejects_bad_arguments_on_the_host(lib):
    def call(logits=0x10000, B=1, S=16, V=1024, tau=0.9, step=1, T=4, masked=0x20000, tokens=0x30000,
             ws=0x40000, ws_bytes=1 << 20):
        return lib.tt_unmask(logits, N.TT_FP32, B, S, V, tau, step, T, masked, tokens, None, None, None,
                             ws, ws_bytes, None, None)
    assert call(step=0) == N.TT_ERR_INVALID_ARG
    assert call(T=0) == N.TT_ERR_INVALID_ARG
    assert call(tau=float("nan")) == N.TT_ERR_INVALID_ARG
    assert call(V=0) == N.TT_ERR_INVALID_ARG
    assert call(masked=0) == N.TT_ERR_INVALID_ARG
    assert call(tokens=0) == N.TT_ERR_INVALID_ARG
    assert call(logits=0) == N.TT_ERR_INVALID_ARG
    assert call(ws=0) == N.TT_ERR_CAPACITY
    assert call(ws_bytes=16) == N.TT_ERR_CAPACITY
    assert call(S=4096) == N.TT_ERR_UNSUPPORTED
    assert call(B=0) == N.TT_OK


def test_masked_nll_and_schedule_reject_bad_arguments_on_the_host(lib):
    n = ctypes.c_size_t(0)
    assert lib.tt_masked_nll_workspace_size(32, 16, 131072, N.TT_BF16, ctypes.byref(n)) == N.TT_OK
    # 4 units of 64 KB per row in blocks of 2: 2 partials of 16 bytes per row, plus tickets
    assert n.value >= 32 * 16 * 2 * 16 + 32 * 4
    assert lib.tt_masked_nll_workspace_size(1, 0, 10, N.TT_BF16, ctypes.byref(n)) == N.TT_ERR_INVALID_ARG
    assert lib.tt_masked_nll_workspace_size(1, 16, 10, 5, ctypes.byref(n)) == N.TT_ERR_INVALID_ARG

    def call(logits=0x10000, dtype=N.TT_BF16, B=2, S=16, V=1024, targets=0x20000, masked=0x30000, ws=0x40000,
             ws_bytes=1 << 20):
        return lib.tt_masked_nll(logits, dtype, B, S, V, targets, masked, None, None, None, ws, ws_bytes, None,
                                 None)
    assert call(targets=0) == N.TT_ERR_INVALID_ARG
    assert call(masked=0) == N.TT_ERR_INVALID_ARG
    assert call(logits=0) == N.TT_ERR_INVALID_ARG
    assert call(V=0) == N.TT_ERR_INVALID_ARG
    assert call(ws=0) == N.TT_ERR_CAPACITY
    assert call(ws_bytes=64) == N.TT_ERR_CAPACITY
    assert call(S=2048) == N.TT_ERR_UNSUPPORTED
    assert call(V=1003) == N.TT_ERR_UNSUPPORTED            # rows not 16-byte aligned
    assert call(logits=0x10002) == N.TT_ERR_UNSUPPORTED
    assert call(B=0) == N.TT_OK
    # the corruption step
    sched = lib.tt_linear_schedule_mask
    assert sched(None, 0, 0x2000, 2, 16, -1, None, 0x3000, None, None) == N.TT_ERR_INVALID_ARG      # no u
    assert sched(None, 0x1000, 0, 2, 16, -1, None, 0x3000, None, None) == N.TT_ERR_INVALID_ARG      # no t
    assert sched(None, 0x1000, 0x2000, 2, 16, -1, None, 0, None, None) == N.TT_ERR_INVALID_ARG      # no mask out
    assert sched(None, 0x1000, 0x2000, 2, 16, -1, 0x4000, 0x3000, None, None) == N.TT_ERR_INVALID_ARG  # noisy, no clean
    assert sched(None, 0x1000, 0x2000, 2, 0, -1, None, 0x3000, None, None) == N.TT_ERR_INVALID_ARG
    assert sched(None, 0, 0, 0, 16, -1, None, 0, None, None) == N.TT_OK                             # empty batch


def test_append_rejects_bad_arguments_on_the_host(lib):
    two = (N.tt_kv_cache * 2)(_cache(), _cache(ctx_len=0x5000))
    kn = N.ptr_array([0x10000, 0x11000])
    vn = N.ptr_array([0x20000, 0x21000])
    assert lib.tt_kv_append(None, 1, kn, vn, None, 1, 16, None, None) == N.TT_ERR_INVALID_ARG
    assert lib.tt_kv_append(two, 0, kn, vn, None, 1, 16, None, None) == N.TT_ERR_INVALID_ARG
    # layers of one call must share their length array
    assert lib.tt_kv_append(two, 2, kn, vn, None, 1, 16, None, None) == N.TT_ERR_INVALID_ARG
    same = (N.tt_kv_cache * 2)(_cache(), _cache(head_dim=64))
    assert lib.tt_kv_append(same, 2, kn, vn, None, 1, 16, None, None) == N.TT_ERR_INVALID_ARG
    assert lib.tt_kv_append(two, 1, N.ptr_array([0]), vn, None, 1, 16, None, None) == N.TT_ERR_INVALID_ARG
    assert lib.tt_kv_append(two, 1, kn, vn, None, 1, 0, None, None) == N.TT_ERR_INVALID_ARG
    assert lib.tt_kv_append(two, 1, kn, vn, None, 1, 1025, None, None) == N.TT_ERR_UNSUPPORTED
    many = (N.tt_kv_cache * 17)(*[_cache() for _ in range(17)])
    kn17, vn17 = N.ptr_array([0x10000] * 17), N.ptr_array([0x20000] * 17)
    assert lib.tt_kv_append(many, 17, kn17, vn17, None, 1, 16, None, None) == N.TT_ERR_UNSUPPORTED
    assert lib.tt_kv_append(two, 1, N.ptr_array([0x10008]), vn, None, 1, 16, None, None) == N.TT_ERR_UNSUPPORTED
    big = (N.tt_kv_cache * 1)(_cache(max_pages_per_seq=(1 << 24) + 1))   # more than 2^30 tokens
    assert lib.tt_kv_append(big, 1, kn, vn, None, 1, 16, None, None) == N.TT_ERR_UNSUPPORTED
    assert lib.tt_kv_append(two, 1, kn, vn, None, 0, 16, None, None) == N.TT_OK


def test_block_step_and_error_word_reject_bad_arguments(lib):
    one = (N.tt_kv_cache * 1)(_cache())
    p = N.ptr_array([0x10000])
    args = dict(B=1, S=16, Hq=32, V=1024, tau=0.9, step=1, T=4)

    def call(ws=0x50000, ws_bytes=1 << 30, step=1, n_layers=1, cache=one):
        return lib.tt_block_step(cache, n_layers, p, p, p, p, 0x60000, args["B"], args["S"], args["Hq"],
                                 args["V"], args["tau"], step, args["T"], 0.1, 0x70000, 0x80000, None, None,
                                 None, ws, ws_bytes, None, None)
    assert call(n_layers=0) == N.TT_ERR_INVALID_ARG
    assert call(cache=None) == N.TT_ERR_INVALID_ARG
    assert call(ws=0) == N.TT_ERR_CAPACITY
    assert call(step=0) == N.TT_ERR_INVALID_ARG
    code = ctypes.c_uint32(0)
    assert lib.tt_get_device_error(None, None, ctypes.byref(code)) == N.TT_ERR_INVALID_ARG
    assert lib.tt_get_device_error(0x1000, None, None) == N.TT_ERR_INVALID_ARG


def test_wait_self_check_rejects_bad_arguments_on_the_host(lib):
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: validation fails first
    assert lib.tt_check_wait_timeout(0, fake, None) == N.TT_ERR_INVALID_ARG
    assert lib.tt_check_wait_timeout((1 << 24) + 1, fake, None) == N.TT_ERR_INVALID_ARG
    assert lib.tt_check_wait_timeout(100, None, None) == N.TT_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch):
    """Without the built library every call raises: there is no fallback implementation."""
    monkeypatch.setattr(N, "_lib", None)
    monkeypatch.setattr(N, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libtt_denoise.so"))
    with pytest.raises(N.NativeLibraryMissing):
        N.lib()


def test_binding_rejects_host_tensors_before_any_call():
    torch = pytest.importorskip("torch")
    from block_wise_diffusion_denoise_b300 import api
    logits = torch.zeros((1, 16, 64), dtype=torch.bfloat16)
    masked = torch.ones((1, 16), dtype=torch.uint8)
    tokens = torch.zeros((1, 16), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.tt_unmask(logits, masked, tokens, 0.9, 1, 4)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.tt_unmask_noalloc(logits, masked, tokens, 0.9, 1, 4)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.KVCache(torch.zeros((2, 1, 64, 128), dtype=torch.bfloat16),
                    torch.zeros((2, 1, 64, 128), dtype=torch.bfloat16),
                    torch.zeros((1, 2), dtype=torch.int32), torch.zeros(1, dtype=torch.int32))
