"""Python binding of libkvc.so (include/kvc.h): argument marshalling only.

The functions below carry the C names and take torch tensors (device memory) and
torch CUDA streams; they pass raw pointers to the library and raise ``KvcError``
on a non-zero return code.  Every step of the computation runs in the library's
CUDA kernels.  ``KVCache`` bundles a handle with torch-allocated buffers.

Importing this module loads libkvc.so and fails loudly if it has not been built
(``python -m diffusion_serving_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "kvc.h")

F32, F16, BF16 = 0, 1, 2
LINEAR, CIRCULAR, PACKED = 0, 1, 2
CAUSAL, KERNEL_SIMT, DETERMINISTIC = 1, 256, 512
OK, ERR_ARG, ERR_UNSUPPORTED, ERR_RANGE, ERR_CUDA, ERR_DEVICE = 0, -1, -2, -3, -4, -5
DEV_BAD_SLOT, DEV_BAD_KVLEN, DEV_BAD_CUSEQ, DEV_OVERFLOW, DEV_NO_CHUNK, DEV_TIMEOUT, DEV_BAD_POS = 1, 2, 4, 8, 16, 32, 64
META_ROW0 = 4

DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
CODE_DTYPE = {v: k for k, v in DTYPE_CODE.items()}
LAYOUT_CODE = {"linear": LINEAR, "circular": CIRCULAR, "packed": PACKED}


class KvcError(RuntimeError):
    def __init__(self, code: int, what: str, bits: int = 0):
        self.code, self.bits = code, bits
        super().__init__(f"{what}: {kvc_strerror(code)} ({code})" + (f", device bits {bits:#x}" if bits else ""))


class kvc_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("sink", ctypes.c_int32), ("window", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("capacity", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("softmax_scale", ctypes.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvc.so is not built ({LIB_PATH}); run python -m diffusion_serving_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, U32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
    cfgp = ctypes.POINTER(kvc_config)
    sig = {
        "kvc_meta_bytes": (SZ, [cfgp]),
        "kvc_workspace_bytes": (SZ, [cfgp]),
        "kvc_create": (ctypes.c_int, [cfgp, P, P, P, P, P, ctypes.POINTER(P)]),
        "kvc_advance": (ctypes.c_int, [P, I32, I32, P]),
        "kvc_write": (ctypes.c_int, [P, P, P, I32, P, P]),
        "kvc_write_rope": (ctypes.c_int, [P, P, P, I32, P, P, I32, P]),
        "kvc_append": (ctypes.c_int, [P, P, P, I32, P]),
        "kvc_append_attend_decode": (ctypes.c_int, [P, P, P, P, P, P]),
        "kvc_set_lengths": (ctypes.c_int, [P, P, P, P]),
        "kvc_attend": (ctypes.c_int, [P, P, P, I32, U32, P]),
        "kvc_attend_lse": (ctypes.c_int, [P, P, P, P, I32, U32, P]),
        "kvc_merge": (ctypes.c_int, [I32, I32, I32, P, P, P, P, P, P, P]),
        "kvc_roll_scratch_bytes": (SZ, [cfgp]),
        "kvc_roll_window": (ctypes.c_int, [P, P, P]),
        "kvc_reset": (ctypes.c_int, [P, I32, P]),
        "kvc_get_error": (ctypes.c_int, [P, P, ctypes.POINTER(I32)]),
        "kvc_destroy": (ctypes.c_int, [P]),
        "kvc_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "kvc_attend_decode_noalloc": (ctypes.c_int, [cfgp, P, P, P, P, P, P]),
        "kvc_lengths_bytes": (SZ, [I32]),
        "kvc_lengths_create": (ctypes.c_int, [I32, I32, I32, P, P, ctypes.POINTER(P)]),
        "kvc_lengths_set": (ctypes.c_int, [P, P, P, P]),
        "kvc_use_lengths": (ctypes.c_int, [P, P]),
        "kvc_lengths_destroy": (ctypes.c_int, [P]),
        "kvc_debug_stall_waits": (ctypes.c_int, [P, ctypes.c_uint64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()


def header_functions() -> list[str]:
    """Names of the functions include/kvc.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(kvc_\w+)\s*\(", text, flags=re.M)


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("kvc: tensors are passed by pointer as dense row-major arrays and must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != OK:
        raise KvcError(rc, what)


def make_config(batch, heads, kv_heads, head_dim, dtype, layout, *, sink=0, window=0, chunk=0,
                capacity=0, softmax_scale=0.0) -> kvc_config:
    d = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    lay = LAYOUT_CODE[layout] if isinstance(layout, str) else int(layout)
    return kvc_config(batch, heads, kv_heads, head_dim, sink, window, chunk, capacity, d, lay, softmax_scale)


# ---------------------------------------------------------------------------
# the C entry points, same names
# ---------------------------------------------------------------------------
def kvc_meta_bytes(cfg: kvc_config) -> int:
    return _lib.kvc_meta_bytes(ctypes.byref(cfg))


def kvc_workspace_bytes(cfg: kvc_config) -> int:
    return _lib.kvc_workspace_bytes(ctypes.byref(cfg))


def kvc_create(cfg: kvc_config, k_store, v_store, meta, workspace=None, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(_lib.kvc_create(ctypes.byref(cfg), _ptr(k_store), _ptr(v_store), _ptr(meta), _ptr(workspace),
                           _stream(stream), ctypes.byref(h)), "kvc_create")
    return h.value


def kvc_advance(h: int, row: int = -1, n_tokens: int = 0, stream=None) -> None:
    _check(_lib.kvc_advance(h, row, n_tokens, _stream(stream)), "kvc_advance")


def kvc_write(h: int, k, v, n_tokens: int, slots=None, stream=None) -> None:
    _check(_lib.kvc_write(h, _ptr(k), _ptr(v), n_tokens, _ptr(slots), _stream(stream)), "kvc_write")


def kvc_append(h: int, k, v, n_tokens: int, stream=None) -> None:
    _check(_lib.kvc_append(h, _ptr(k), _ptr(v), n_tokens, _stream(stream)), "kvc_append")


def kvc_append_attend_decode(h: int, k_new, v_new, q, out, stream=None) -> None:
    _check(_lib.kvc_append_attend_decode(h, _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out), _stream(stream)),
           "kvc_append_attend_decode")


def kvc_write_rope(h: int, k, v, n_tokens: int, rope, rope_positions: int, slots=None, stream=None) -> None:
    _check(_lib.kvc_write_rope(h, _ptr(k), _ptr(v), n_tokens, _ptr(slots), _ptr(rope), rope_positions,
                               _stream(stream)), "kvc_write_rope")


def kvc_set_lengths(h: int, kv_len=None, cu_seqlens=None, stream=None) -> None:
    _check(_lib.kvc_set_lengths(h, _ptr(kv_len), _ptr(cu_seqlens), _stream(stream)), "kvc_set_lengths")


def kvc_attend(h: int, q, out, n_q: int, flags: int = 0, stream=None) -> None:
    _check(_lib.kvc_attend(h, _ptr(q), _ptr(out), n_q, flags, _stream(stream)), "kvc_attend")


def kvc_attend_lse(h: int, q, out, lse, n_q: int, flags: int = 0, stream=None) -> None:
    _check(_lib.kvc_attend_lse(h, _ptr(q), _ptr(out), _ptr(lse), n_q, flags, _stream(stream)), "kvc_attend_lse")


def kvc_merge(dtype, n_rows: int, head_dim: int, o_a, lse_a, o_b, lse_b, out, lse_out=None, stream=None) -> None:
    d = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    _check(_lib.kvc_merge(d, n_rows, head_dim, _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(out),
                          _ptr(lse_out), _stream(stream)), "kvc_merge")


def kvc_roll_scratch_bytes(cfg: kvc_config) -> int:
    return _lib.kvc_roll_scratch_bytes(ctypes.byref(cfg))


def kvc_roll_window(h: int, scratch, stream=None) -> None:
    _check(_lib.kvc_roll_window(h, _ptr(scratch), _stream(stream)), "kvc_roll_window")


def kvc_reset(h: int, row: int = -1, stream=None) -> None:
    _check(_lib.kvc_reset(h, row, _stream(stream)), "kvc_reset")


def kvc_get_error(h: int, stream=None) -> int:
    """Return the device error bits (0 if none) and clear them."""
    bits = ctypes.c_int32(0)
    rc = _lib.kvc_get_error(h, _stream(stream), ctypes.byref(bits))
    if rc not in (OK, ERR_DEVICE):
        raise KvcError(rc, "kvc_get_error")
    return bits.value


def kvc_destroy(h: int) -> None:
    _check(_lib.kvc_destroy(h), "kvc_destroy")


def kvc_strerror(code: int) -> str:
    return _lib.kvc_strerror(code).decode()


def _check_noalloc_args(cfg: kvc_config, k_store, v_store, meta, q, out):
    """The C call reads and writes through these pointers with sizes taken from cfg, so a
    tensor smaller than cfg says, or of another type, is refused here."""
    dt = CODE_DTYPE.get(cfg.dtype)
    want = (cfg.batch, 1, cfg.heads, cfg.head_dim)
    for name, t in (("q", q), ("out", out)):
        if tuple(t.shape) != want or t.dtype != dt:
            raise ValueError(f"kvc: {name} must be {list(want)} {dt}, got {list(t.shape)} {t.dtype}")
    rows = {LINEAR: cfg.batch * cfg.capacity, CIRCULAR: cfg.batch * cfg.window, PACKED: cfg.capacity}.get(cfg.layout, 0)
    need = rows * cfg.kv_heads * cfg.head_dim
    for name, t in (("k_store", k_store), ("v_store", v_store)):
        if t.dtype != dt or t.numel() < need:
            raise ValueError(f"kvc: {name} must hold {need} {dt} elements, got {t.numel()} {t.dtype}")
    mb = kvc_meta_bytes(cfg)
    if meta.dtype != torch.int32 or meta.numel() * 4 < mb:
        raise ValueError(f"kvc: meta must be int32 of at least {mb} bytes, got {meta.numel()} {meta.dtype}")


def kvc_attend_decode_noalloc(cfg: kvc_config, k_store, v_store, meta, q, out, stream=None) -> None:
    """Decode attention for callers that cannot allocate device memory (see kvc.h)."""
    _check_noalloc_args(cfg, k_store, v_store, meta, q, out)
    _check(_lib.kvc_attend_decode_noalloc(ctypes.byref(cfg), _ptr(k_store), _ptr(v_store), _ptr(meta), _ptr(q),
                                          _ptr(out), _stream(stream)), "kvc_attend_decode_noalloc")


def kvc_debug_stall_waits(h: int, ns: int) -> None:
    """Testing hook: the handle's later attends wait ns nanoseconds on a barrier nothing
    signals, then give up (KVC_DEV_TIMEOUT); 0 turns it off."""
    _check(_lib.kvc_debug_stall_waits(h, ns), "kvc_debug_stall_waits")


def kvc_lengths_bytes(batch: int) -> int:
    return _lib.kvc_lengths_bytes(batch)


def kvc_lengths_create(batch: int, layout, capacity: int, block, stream=None) -> int:
    lay = LAYOUT_CODE[layout] if isinstance(layout, str) else int(layout)
    h = ctypes.c_void_p()
    _check(_lib.kvc_lengths_create(batch, lay, capacity, _ptr(block), _stream(stream), ctypes.byref(h)),
           "kvc_lengths_create")
    return h.value


def kvc_lengths_set(L: int, kv_len=None, cu_seqlens=None, stream=None) -> None:
    _check(_lib.kvc_lengths_set(L, _ptr(kv_len), _ptr(cu_seqlens), _stream(stream)), "kvc_lengths_set")


def kvc_use_lengths(h: int, L) -> None:
    _check(_lib.kvc_use_lengths(h, L), "kvc_use_lengths")


def kvc_lengths_destroy(L: int) -> None:
    _check(_lib.kvc_lengths_destroy(L), "kvc_lengths_destroy")


# ---------------------------------------------------------------------------
# convenience owners of the device buffers
# ---------------------------------------------------------------------------
class KVLengths:
    """A shared length layout (kv_len per row, or packed cu_seqlens) over a torch-allocated
    block; handles point at it with ``KVCache.use_lengths``."""

    def __init__(self, batch, layout, capacity, device="cuda", stream=None):
        self.batch = batch
        nbytes = kvc_lengths_bytes(batch)
        self.block = torch.zeros(nbytes // 4, dtype=torch.int32, device=device)
        self.handle = kvc_lengths_create(batch, layout, capacity, self.block, stream)

    def set(self, kv_len=None, cu_seqlens=None, stream=None):
        kvc_lengths_set(self.handle, kv_len, cu_seqlens, stream)

    def close(self):
        if self.handle:
            kvc_lengths_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

class KVCache:
    """A kvc handle plus torch-allocated K/V stores, meta block and workspace."""

    def __init__(self, batch, heads, kv_heads, head_dim, dtype, layout, *, sink=0, window=0, chunk=0,
                 capacity=0, softmax_scale=0.0, device="cuda", stream=None):
        self.cfg = make_config(batch, heads, kv_heads, head_dim, dtype, layout, sink=sink, window=window,
                               chunk=chunk, capacity=capacity, softmax_scale=softmax_scale)
        self.dtype = dtype
        self.layout = LAYOUT_CODE[layout] if isinstance(layout, str) else int(layout)
        slots = window if self.layout == CIRCULAR else capacity
        shape = (slots, kv_heads, head_dim) if self.layout == PACKED else (batch, slots, kv_heads, head_dim)
        self.k_store = torch.empty(shape, dtype=dtype, device=device)
        self.v_store = torch.empty(shape, dtype=dtype, device=device)
        mb = kvc_meta_bytes(self.cfg)
        if mb == 0:
            raise KvcError(ERR_ARG, "kvc_meta_bytes")
        self.meta = torch.zeros(mb // 4, dtype=torch.int32, device=device)
        wb = kvc_workspace_bytes(self.cfg)
        self.workspace = torch.zeros(max(wb, 16) // 4, dtype=torch.int32, device=device)
        self.handle = kvc_create(self.cfg, self.k_store, self.v_store, self.meta, self.workspace, stream)

    def advance(self, row=-1, n_tokens=None, stream=None):
        kvc_advance(self.handle, row, self.cfg.chunk if n_tokens is None else n_tokens, stream)

    def _check_rows(self, what, t, heads):
        """t must be [batch, n, heads, head_dim] in the store's dtype."""
        shape = (self.cfg.batch, heads, self.cfg.head_dim)
        if t.dim() != 4 or (t.shape[0], t.shape[2], t.shape[3]) != shape or t.dtype != self.dtype:
            raise ValueError(f"kvc: {what} must be [{shape[0]}, n, {shape[1]}, {shape[2]}] {self.dtype}, "
                             f"got {list(t.shape)} {t.dtype}")

    def _check_kv(self, k, v):
        self._check_rows("k", k, self.cfg.kv_heads)
        self._check_rows("v", v, self.cfg.kv_heads)
        if k.shape != v.shape:
            raise ValueError(f"kvc: k {list(k.shape)} and v {list(v.shape)} differ")

    def _check_q(self, q, out):
        self._check_rows("q", q, self.cfg.heads)
        if out.shape != q.shape or out.dtype != q.dtype:
            raise ValueError(f"kvc: out must match q ({list(q.shape)} {q.dtype})")

    def write(self, k, v, slots=None, stream=None):
        self._check_kv(k, v)
        kvc_write(self.handle, k, v, k.shape[1], slots, stream)

    def append(self, k, v, stream=None):
        """Reserve k.shape[1] slots after those filled (LINEAR) and write k, v there."""
        self._check_kv(k, v)
        kvc_append(self.handle, k, v, k.shape[1], stream)

    def append_attend(self, k, v, q, out=None, stream=None):
        """One decode step in one launch: append one token per row (k, v [B, 1, Hkv, D])
        and attend q [B, 1, H, D] over the prefix with it (LINEAR, 16-bit)."""
        self._check_kv(k, v)
        if k.shape[1] != 1 or q.shape[1] != 1:
            raise ValueError("kvc: append_attend takes one new token and one query per row")
        if out is None:
            out = torch.empty_like(q)
        self._check_q(q, out)
        kvc_append_attend_decode(self.handle, k, v, q, out, stream)
        return out

    def write_rope(self, k, v, rope, slots=None, stream=None):
        """Write with K rotated by the (cos, sin) table ``rope`` [positions, D/2, 2] fp32."""
        self._check_kv(k, v)
        kvc_write_rope(self.handle, k, v, k.shape[1], rope, rope.shape[0], slots, stream)

    def set_lengths(self, kv_len=None, cu_seqlens=None, stream=None):
        kvc_set_lengths(self.handle, kv_len, cu_seqlens, stream)

    def use_lengths(self, lengths: "KVLengths | None"):
        """Read lengths from a shared layout (None: from this handle's own meta block).
        The layout object is kept referenced so that it outlives this use."""
        kvc_use_lengths(self.handle, None if lengths is None else lengths.handle)
        self.shared_lengths = lengths

    def attend(self, q, out=None, flags=0, stream=None):
        if out is None:
            out = torch.empty_like(q)
        self._check_q(q, out)
        kvc_attend(self.handle, q, out, q.shape[1], flags, stream)
        return out

    def attend_lse(self, q, out=None, flags=0, stream=None):
        """(out, lse) with lse [B, n_q, H] fp32."""
        if out is None:
            out = torch.empty_like(q)
        self._check_q(q, out)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
        kvc_attend_lse(self.handle, q, out, lse, q.shape[1], flags, stream)
        return out, lse

    def reset(self, row=-1, stream=None):
        kvc_reset(self.handle, row, stream)

    def get_error(self, stream=None) -> int:
        return kvc_get_error(self.handle, stream)

    def row_state(self):
        """(chunks, first slot, filled, kv_len) per row, read from the meta block."""
        m = self.meta[META_ROW0:META_ROW0 + 4 * self.cfg.batch].view(self.cfg.batch, 4)
        return m.cpu().tolist()

    def close(self):
        if self.handle:
            kvc_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
