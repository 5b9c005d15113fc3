"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
sizes its buffers and rejects bad configs before touching the device."""
import ctypes
import os
import subprocess

import pytest

from diffusion_serving_gb300 import kvc


def test_library_exports_every_declared_function():
    names = kvc.header_functions()
    assert len(names) == 25
    for n in names:
        assert hasattr(kvc._lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", kvc.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported


def test_library_has_no_torch_dependency():
    out = subprocess.run(["ldd", kvc.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_header_compiles_as_c():
    src = os.path.join(os.path.dirname(kvc.HEADER_PATH), "kvc.h")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", src],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_config_struct_layout():
    assert ctypes.sizeof(kvc.kvc_config) == 44


def cfg(**kw):
    base = dict(batch=2, heads=12, kv_heads=12, head_dim=128, dtype=kvc.BF16, layout="circular",
                sink=4680, window=32760, chunk=4680)
    base.update(kw)
    return kvc.make_config(base.pop("batch"), base.pop("heads"), base.pop("kv_heads"), base.pop("head_dim"),
                           base.pop("dtype"), base.pop("layout"), **base)


def test_meta_bytes():
    # 4 header words + 4 per row + B + 1 cu_seqlens words, rounded up to 256 bytes
    assert kvc.kvc_meta_bytes(cfg()) == 256
    big = cfg(batch=100)
    assert kvc.kvc_meta_bytes(big) == ((4 + 400 + 101) * 4 + 255) // 256 * 256


@pytest.mark.parametrize("bad", [dict(heads=12, kv_heads=5), dict(head_dim=96), dict(sink=100),
                                 dict(window=4680), dict(dtype=7), dict(batch=0), dict(chunk=0),
                                 dict(layout="linear", capacity=0), dict(softmax_scale=-1.0)])
def test_bad_configs_are_rejected_on_the_host(bad):
    c = cfg(**bad)
    assert kvc.kvc_meta_bytes(c) == 0
    assert kvc.kvc_workspace_bytes(c) == 0
    h = ctypes.c_void_p()
    rc = kvc._lib.kvc_create(ctypes.byref(c), 16, 16, 16, 16, None, ctypes.byref(h))
    assert rc in (kvc.ERR_ARG, kvc.ERR_UNSUPPORTED)
    assert h.value is None


def test_misaligned_store_is_rejected():
    h = ctypes.c_void_p()
    assert kvc._lib.kvc_create(ctypes.byref(cfg()), 8, 16, 16, 16, None, ctypes.byref(h)) == kvc.ERR_ARG


def test_workspace_only_for_split_decode():
    assert kvc.kvc_workspace_bytes(cfg(dtype=kvc.F32)) == 0
    dec = cfg(batch=1, heads=32, kv_heads=8, layout="linear", capacity=32768, dtype=kvc.F16)
    n = kvc.kvc_workspace_bytes(dec)
    assert n > 0 and n % 256 == 0


def test_null_handle_calls_fail_cleanly():
    assert kvc._lib.kvc_advance(None, -1, 1, None) == kvc.ERR_ARG
    assert kvc._lib.kvc_attend(None, None, None, 1, 0, None) == kvc.ERR_ARG
    assert kvc._lib.kvc_reset(None, -1, None) == kvc.ERR_ARG
    assert kvc._lib.kvc_get_error(None, None, None) == kvc.ERR_ARG
    assert kvc._lib.kvc_append_attend_decode(None, None, None, None, None, None) == kvc.ERR_ARG
    assert kvc.kvc_strerror(kvc.ERR_RANGE) == "length out of range"


def test_binding_rejects_strided_tensors():
    """The C ABI takes dense row-major arrays: the binding refuses a view with other strides."""
    import torch
    with pytest.raises(ValueError):
        kvc._ptr(torch.empty(4, 8).t())
    with pytest.raises(ValueError):
        kvc._ptr(torch.empty(2, 6, 4, 8)[:, ::2])
    assert kvc._ptr(torch.empty(2, 3, 4, 8)) != 0
    assert kvc._ptr(None) is None


def test_binding_refuses_mismatched_noalloc_buffers():
    """kvc_attend_decode_noalloc takes only pointers; its wrapper checks the tensors
    against the config before any call, so a wrong q / out shape or type, an undersized
    store or meta block never reaches the library (no device is needed for this)."""
    import torch
    c = kvc.make_config(2, 8, 2, 64, torch.float16, "linear", capacity=32)
    store = torch.zeros(2 * 32 * 2 * 64, dtype=torch.float16)
    meta = torch.zeros(kvc.kvc_meta_bytes(c) // 4, dtype=torch.int32)
    q = torch.zeros(2, 1, 8, 64, dtype=torch.float16)
    bad = {
        "q shape": dict(q=torch.zeros(2, 2, 8, 64, dtype=torch.float16)),
        "q dtype": dict(q=torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16)),
        "out shape": dict(out=torch.zeros(2, 1, 4, 64, dtype=torch.float16)),
        "store size": dict(k_store=store[:-1]),
        "store dtype": dict(v_store=torch.zeros(2 * 32 * 2 * 64, dtype=torch.float32)),
        "meta size": dict(meta=meta[:-1]),
        "meta dtype": dict(meta=torch.zeros(64, dtype=torch.float32)),
    }
    for what, change in bad.items():
        args = dict(k_store=store, v_store=store, meta=meta, q=q, out=q.clone())
        args.update(change)
        with pytest.raises(ValueError):
            kvc._check_noalloc_args(c, **args)
    kvc._check_noalloc_args(c, store, store, meta, q, q.clone())      # the matching set passes


def test_shared_lengths_host_checks():
    """Length layouts: sizes and the host-side refusals, before any device work."""
    assert kvc.kvc_lengths_bytes(0) == 0
    assert kvc.kvc_lengths_bytes(2) == kvc.kvc_meta_bytes(cfg(batch=2, layout="packed", capacity=64))
    h = ctypes.c_void_p()
    assert kvc._lib.kvc_lengths_create(2, kvc.CIRCULAR, 64, 256, None, ctypes.byref(h)) == kvc.ERR_UNSUPPORTED
    assert kvc._lib.kvc_lengths_create(0, kvc.PACKED, 64, 256, None, ctypes.byref(h)) == kvc.ERR_ARG
    assert kvc._lib.kvc_lengths_create(2, kvc.PACKED, 64, 8, None, ctypes.byref(h)) == kvc.ERR_ARG   # misaligned
    assert kvc._lib.kvc_lengths_create(2, kvc.PACKED, 64, None, None, ctypes.byref(h)) == kvc.ERR_ARG
    assert kvc._lib.kvc_lengths_set(None, 16, None, None) == kvc.ERR_ARG
    assert kvc._lib.kvc_use_lengths(None, None) == kvc.ERR_ARG
