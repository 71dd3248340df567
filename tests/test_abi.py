"""The C ABI library builds for sm_103a, loads, exports every function
include/infllmv2.h declares, and rejects bad arguments on the host -- all
without a GPU (no call here reaches a kernel launch)."""
import ctypes

import pytest

from block_sparse_long_infllm_gb300 import infllmv2


def test_exports_every_declared_function(built_lib):
    names = infllmv2.declared_functions()
    assert {"infllmv2_kernel_pool", "infllmv2_append", "infllmv2_block_select", "infllmv2_sparse_attn_fwd",
            "infllmv2_decode", "infllmv2_sparse_attn_bwd", "infllmv2_decode_host"} <= set(names)
    for n in names:
        assert hasattr(built_lib, n), n


def test_status_strings_and_version(built_lib):
    assert infllmv2.status_string(0) == "ok"
    for code in range(-7, 0):
        assert infllmv2.status_string(code) not in ("", "unknown status")
    assert infllmv2.status_string(12345) == "unknown status"
    assert infllmv2.version() >= 100


P = dict(block_size=64, kernel_size=32, kernel_stride=16, topk=64, n_init_blocks=1,
         n_local_blocks=2, dense_len=8192)


def test_selection_capacity(built_lib):
    assert infllmv2.selection_capacity(dict(P, dense_len=0), 131072) == 64 + 1 + 2
    # below dense_len every causal block may be chosen: ceil(8191 / 64) = 128 blocks
    assert infllmv2.selection_capacity(P, 131072) == 128
    assert infllmv2.selection_capacity(dict(P, topk=200), 131072) == 203
    # never more than the cache holds
    assert infllmv2.selection_capacity(dict(P, dense_len=0), 1000) == 16
    assert infllmv2.selection_capacity(dict(P, n_local_blocks=0), 1000) == -1
    assert infllmv2.selection_capacity(dict(P, block_size=96), 1000) == -1


def test_workspace_sizes(built_lib):
    sel = infllmv2.workspace_size(infllmv2.ENTRY_BLOCK_SELECT, 1, 4096, 32, 2, 128, 32768,
                                  dict(P, block_size=128))
    assert sel >= 2 * 4096 * 256 * 4
    dec = infllmv2.workspace_size(infllmv2.ENTRY_DECODE, 4, 1, 32, 2, 128, 131072, P)
    assert dec > 4 * 2 * 2048 * 4
    assert infllmv2.workspace_size(infllmv2.ENTRY_DECODE, 4, 1, 32, 2, 96, 131072, P) == 0
    assert infllmv2.workspace_size(99, 4, 1, 32, 2, 128, 131072, P) == 0


def _params(**kw):
    return ctypes.byref(infllmv2.Params.make(dict(P, **kw)))


@pytest.mark.parametrize("kw,code", [
    (dict(block_size=32), infllmv2.ERR_UNSUPPORTED),
    (dict(n_local_blocks=0), infllmv2.ERR_INVALID_ARG),
    (dict(kernel_stride=0), infllmv2.ERR_INVALID_ARG),
    (dict(topk=-1), infllmv2.ERR_INVALID_ARG),
    (dict(kernel_size=200), infllmv2.ERR_UNSUPPORTED),
])
def test_bad_params_rejected_on_host(built_lib, kw, code):
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the check fails first
    rc = built_lib.infllmv2_kernel_pool(fake, fake, 1, 2, 4096, 255, 128, 0, 4096, _params(**kw), None)
    assert rc == code


def test_bad_shapes_rejected_on_host(built_lib):
    fake = ctypes.c_void_p(1 << 20)
    lib = built_lib
    # d outside {64, 128}
    assert lib.infllmv2_block_select(fake, fake, fake, 1, 1, 32, 2, 96, 4096, 255, fake, fake, 67, fake,
                                     1 << 30, _params(), None) == infllmv2.ERR_UNSUPPORTED
    # group size 3
    assert lib.infllmv2_block_select(fake, fake, fake, 1, 1, 6, 2, 128, 4096, 255, fake, fake, 67, fake,
                                     1 << 30, _params(), None) == infllmv2.ERR_UNSUPPORTED
    # S_max below the selection capacity
    assert lib.infllmv2_block_select(fake, fake, fake, 1, 1, 32, 2, 128, 4096, 255, fake, fake, 10, fake,
                                     1 << 30, _params(dense_len=0), None) == infllmv2.ERR_INVALID_ARG
    # workspace too small
    assert lib.infllmv2_block_select(fake, fake, fake, 1, 1, 32, 2, 128, 4096, 255, fake, fake, 67, fake,
                                     16, _params(dense_len=0), None) == infllmv2.ERR_WORKSPACE
    # misaligned pointer
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert lib.infllmv2_sparse_attn_fwd(odd, fake, fake, None, None, 0, fake, 1, 8, 32, 2, 128, 4096, fake,
                                        None, None, 0, _params(), None) == infllmv2.ERR_INVALID_ARG
    # more queries than the cache holds
    assert lib.infllmv2_sparse_attn_fwd(fake, fake, fake, None, None, 0, fake, 1, 5000, 32, 2, 128, 4096,
                                        fake, None, None, 0, _params(), None) == infllmv2.ERR_INVALID_ARG
    # decode: several drafts need a tree mask; more than 64 drafts do not fit a uint64
    assert lib.infllmv2_decode(fake, fake, fake, fake, fake, None, None, None, 1, 2, 32, 2, 128, 4096, 255,
                               fake, None, None, None, 0, fake, 1 << 30, _params(), None) == infllmv2.ERR_INVALID_ARG
    assert lib.infllmv2_decode(fake, fake, fake, fake, fake, fake, fake, fake, 1, 65, 32, 2, 128, 4096, 255,
                               fake, None, None, None, 0, fake, 1 << 30, _params(), None) == infllmv2.ERR_UNSUPPORTED
    # kernel pool range past the cache
    assert lib.infllmv2_kernel_pool(fake, fake, 1, 2, 4096, 255, 128, 0, 4097, _params(), None) == \
        infllmv2.ERR_INVALID_ARG
    assert lib.infllmv2_kernel_pool(fake, fake, 1, 2, 4096, 100, 128, 0, 4096, _params(), None) == \
        infllmv2.ERR_INVALID_ARG
    # append: d outside {64, 128}; a missing kernel cache while kernels exist; misaligned K
    assert lib.infllmv2_append(fake, fake, fake, fake, fake, fake, 1, 2, 96, 4096, 255, _params(), None) == \
        infllmv2.ERR_UNSUPPORTED
    assert lib.infllmv2_append(fake, fake, fake, fake, None, fake, 1, 2, 128, 4096, 255, _params(), None) == \
        infllmv2.ERR_INVALID_ARG
    assert lib.infllmv2_append(odd, fake, fake, fake, fake, fake, 1, 2, 128, 4096, 255, _params(), None) == \
        infllmv2.ERR_INVALID_ARG


def test_empty_calls_are_noops(built_lib):
    fake = ctypes.c_void_p(1 << 20)
    assert built_lib.infllmv2_sparse_attn_fwd(fake, fake, fake, None, None, 0, fake, 0, 8, 32, 2, 128, 4096,
                                              fake, None, None, 0, _params(), None) == 0
    assert built_lib.infllmv2_kernel_pool(fake, fake, 1, 2, 4096, 255, 128, 100, 100, _params(), None) == 0
    assert built_lib.infllmv2_append(fake, fake, fake, fake, fake, fake, 0, 2, 128, 4096, 255, _params(), None) == 0


def test_decode_host_checks_before_enqueueing(built_lib):
    fake = ctypes.c_void_p(1 << 20)
    lib = built_lib
    args = dict(B=1, Hq=32, Hkv=2, d=128, L_max=4096, M_max=255)

    def call(q_h=fake, kv_h=fake, o_h=fake, lse_h=None, q_d=fake, kv_d=fake, o_d=fake, lse_d=None, ws_bytes=1 << 30,
             B=1, d=128, params=None):
        return lib.infllmv2_decode_host(q_h, kv_h, o_h, lse_h, q_d, kv_d, o_d, lse_d, fake, fake, fake, B,
                                        args["Hq"], args["Hkv"], d, args["L_max"], args["M_max"], fake, ws_bytes,
                                        params or _params(), None)
    assert call(B=0) == 0                                           # nothing to do
    assert call(lse_h=fake) == infllmv2.ERR_INVALID_ARG             # lse wanted on the host, no device buffer
    assert call(q_h=None) == infllmv2.ERR_INVALID_ARG               # missing host query
    assert call(o_d=None) == infllmv2.ERR_INVALID_ARG               # missing device output
    assert call(q_d=ctypes.c_void_p((1 << 20) + 4)) == infllmv2.ERR_INVALID_ARG  # misaligned staging buffer
    assert call(ws_bytes=16) == infllmv2.ERR_WORKSPACE
    assert call(d=96) == infllmv2.ERR_UNSUPPORTED
    assert call(params=_params(topk=-1)) == infllmv2.ERR_INVALID_ARG


def test_host_memory_direct_checks_its_argument(built_lib):
    assert built_lib.infllmv2_host_memory_direct(None) == infllmv2.ERR_INVALID_ARG


def test_decode_host_binding_checks_types_and_sizes():
    """The binding refuses staging tensors whose type or size would make the C call copy past them
    (checked before any pointer is taken, so CPU tensors stand in here)."""
    torch = pytest.importorskip("torch")
    B, Hq, d = 2, 32, 128
    good = dict(q_host=torch.empty((B, Hq, d), dtype=torch.bfloat16),
                kv_len_host=torch.empty(B, dtype=torch.int32),
                o_host=torch.empty((B, Hq, d), dtype=torch.bfloat16),
                q_dev=torch.empty((B, Hq, d), dtype=torch.bfloat16),
                kv_len_dev=torch.empty(B, dtype=torch.int32),
                o_dev=torch.empty((B, Hq, d), dtype=torch.bfloat16),
                lse_host=torch.empty((B, Hq), dtype=torch.float32),
                lse_dev=torch.empty((B, Hq), dtype=torch.float32))
    infllmv2._check_host_step_buffers(Hkv=2, **good)
    bad_cases = [("o_host", torch.empty((B, Hq, d), dtype=torch.float32)),
                 ("q_dev", torch.empty((B, Hq, d // 2), dtype=torch.bfloat16)),
                 ("kv_len_host", torch.empty(B, dtype=torch.int64)),
                 ("kv_len_dev", torch.empty(B + 1, dtype=torch.int32)),
                 ("lse_host", torch.empty((B, Hq), dtype=torch.float16)),
                 ("lse_dev", None)]
    for name, t in bad_cases:
        with pytest.raises(ValueError):
            infllmv2._check_host_step_buffers(Hkv=2, **dict(good, **{name: t}))
    with pytest.raises(ValueError):
        infllmv2._check_host_step_buffers(Hkv=3, **good)
