"""Python binding of libgdn.so, the GB300 Gated DeltaNet layer core.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/gdn.h``. PyTorch provides
device memory and streams. The binding raises if the library is missing; it
never falls back to another implementation.

Entry points (same names as the C ABI): ``gdn_conv``, ``gdn_seq``,
``gdn_decode``, ``gdn_prefill``, ``gdn_spec_verify``, ``gdn_spec_step``, ``gdn_spec_slots``,
``gdn_chunk_prefill``, ``gdn_chunk_prefill_noalloc``, ``gdn_page_to_slots``, ``gdn_slots_to_page``,
``gdn_chunk_prefill_workspace_bytes``, ``gdn_page_layout``,
``gdn_slot_layout``, ``gdn_check_bounded_wait``, ``gdn_strerror``,
``gdn_abi_version``.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libgdn.so")

GDN_F32 = 0
GDN_BF16 = 1
GDN_REQ_FRESH = 0x1
GDN_REQ_SPEC = 0x2
GDN_REQ_PARITY = 0x4

STATUS = {
    0: "GDN_OK", -1: "GDN_ERR_INVALID_ARG", -2: "GDN_ERR_UNSUPPORTED", -3: "GDN_ERR_LAUNCH",
    -4: "GDN_ERR_WORKSPACE", -5: "GDN_ERR_NO_DEVICE", 1: "GDN_DEV_BAD_PAGE",
    2: "GDN_DEV_BAD_ROWS", 3: "GDN_DEV_BAD_ACCEPTED", 4: "GDN_DEV_STALE_STEP",
    5: "GDN_DEV_TOO_MANY_CANDIDATES", 6: "GDN_DEV_RECORD_OPEN", 7: "GDN_DEV_BAD_FLAG",
    8: "GDN_DEV_TIMEOUT",
}
CODES = {v: k for k, v in STATUS.items()}


class GdnError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({gdn_strerror(code)})")


class Dims(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_width", ctypes.c_int32), ("max_candidates", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32)]

    @property
    def C(self):
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


class Params(ctypes.Structure):
    _fields_ = [("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("conv_bias", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("gate_mode", ctypes.c_int32)]


class Batch(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_rows", ctypes.c_int32),
                ("max_rows", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("row_start", ctypes.c_void_p), ("row_len", ctypes.c_void_p),
                ("page", ctypes.c_void_p), ("flags", ctypes.c_void_p),
                ("n_accepted", ctypes.c_void_p), ("order", ctypes.c_void_p)]


class PageLayout(ctypes.Structure):
    _fields_ = [("page_bytes", ctypes.c_size_t), ("window_offset", ctypes.c_size_t),
                ("window_bytes", ctypes.c_size_t), ("state_offset", ctypes.c_size_t),
                ("state_bytes", ctypes.c_size_t), ("record_offset", ctypes.c_size_t),
                ("record_bytes", ctypes.c_size_t), ("flag_offset", ctypes.c_size_t)]


class SlotLayout(ctypes.Structure):
    _fields_ = [("pool_bytes", ctypes.c_size_t), ("slot_bytes", ctypes.c_size_t),
                ("state_offset", ctypes.c_size_t), ("window_offset", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgdn.so (raises if it was not built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        D, B, PR = ctypes.POINTER(Dims), ctypes.POINTER(Batch), ctypes.POINTER(Params)
        sig = {
            "gdn_page_layout": ([D, ctypes.POINTER(PageLayout)], I),
            "gdn_slot_layout": ([D, ctypes.POINTER(SlotLayout)], I),
            "gdn_conv": ([D, B, PR, P, P, P, I, P, P, P], I),
            "gdn_seq": ([D, B, PR, P, P, P, P, P, P, P], I),
            "gdn_spec_verify": ([D, B, PR, P, P, P, P, P, P, P], I),
            "gdn_spec_step": ([D, B, PR, P, P, P, P, P, P, P, P], I),
            "gdn_decode": ([D, B, PR, P, P, P, P, P, P, P, P], I),
            "gdn_prefill": ([D, B, PR, P, P, P, P, P, I, P, S, P, P], I),
            "gdn_spec_slots": ([D, B, PR, P, P, P, P, P, P, P, P, P], I),
            "gdn_page_to_slots": ([D, I, P, P, I, I, P, P, P, P], I),
            "gdn_slots_to_page": ([D, I, P, P, P, I, I, P, P, P, P], I),
            "gdn_chunk_prefill_workspace_bytes": ([D, B], S),
            "gdn_chunk_prefill": ([D, B, PR, P, P, P, P, P, P, S, P, P], I),
            "gdn_chunk_prefill_noalloc": ([D, B, PR, P, P, P, P, P, P, P], I),
            "gdn_check_bounded_wait": ([ctypes.c_int64, P, P], I),
            "gdn_strerror": ([I], ctypes.c_char_p),
            "gdn_abi_version": ([], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


# ------------------------------------------------------------- marshalling

def _ptr(t):
    """Device/host address of a torch tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, where):
    if code != 0:
        raise GdnError(code, where)


def make_dims(Hk, Hv, Dk, Dv, W=4, Kc=0, io=GDN_BF16, state=GDN_F32, out=GDN_BF16) -> Dims:
    return Dims(Hk, Hv, Dk, Dv, W, Kc, io, state, out)


def make_params(A_log, dt_bias, conv_bias=None, scale=0.0, norm_eps=1e-6, gate_mode=0) -> Params:
    return Params(_ptr(A_log), _ptr(dt_bias), _ptr(conv_bias), float(scale), float(norm_eps),
                  int(gate_mode))


def make_batch(num_requests, num_rows, max_rows, num_pages, row_start, row_len, page, flags,
               n_accepted=None, order=None) -> Batch:
    """Row map from device int32 tensors (flags may be int32 or uint32 bits)."""
    return Batch(int(num_requests), int(num_rows), int(max_rows), int(num_pages), _ptr(row_start),
                 _ptr(row_len), _ptr(page), _ptr(flags), _ptr(n_accepted), _ptr(order))


def gdn_page_layout(dims: Dims) -> PageLayout:
    out = PageLayout()
    _check(load_library().gdn_page_layout(ctypes.byref(dims), ctypes.byref(out)), "gdn_page_layout")
    return out


def gdn_slot_layout(dims: Dims) -> SlotLayout:
    out = SlotLayout()
    _check(load_library().gdn_slot_layout(ctypes.byref(dims), ctypes.byref(out)), "gdn_slot_layout")
    return out


def gdn_conv(dims, batch, params, x, conv_w, y, y_dtype, pages, status, stream=None):
    _check(load_library().gdn_conv(ctypes.byref(dims), ctypes.byref(batch), ctypes.byref(params),
                                   _ptr(x), _ptr(conv_w), _ptr(y), int(y_dtype), _ptr(pages),
                                   _ptr(status), _stream(stream)), "gdn_conv")


def gdn_seq(dims, batch, params, qkv, a, b, o, pages, status, stream=None):
    _check(load_library().gdn_seq(ctypes.byref(dims), ctypes.byref(batch), ctypes.byref(params),
                                  _ptr(qkv), _ptr(a), _ptr(b), _ptr(o), _ptr(pages), _ptr(status),
                                  _stream(stream)), "gdn_seq")


def gdn_decode(dims, batch, params, x, conv_w, a, b, o, pages, status, stream=None):
    _check(load_library().gdn_decode(ctypes.byref(dims), ctypes.byref(batch), ctypes.byref(params),
                                     _ptr(x), _ptr(conv_w), _ptr(a), _ptr(b), _ptr(o), _ptr(pages),
                                     _ptr(status), _stream(stream)), "gdn_decode")


def gdn_prefill(dims, batch, params, qkv, a, b, o, pages, status, chunk_min_rows=0, stream=None,
                workspace=None, workspace_bytes=0):
    _check(load_library().gdn_prefill(ctypes.byref(dims), ctypes.byref(batch), ctypes.byref(params),
                                      _ptr(qkv), _ptr(a), _ptr(b), _ptr(o), _ptr(pages),
                                      int(chunk_min_rows), _ptr(workspace), int(workspace_bytes),
                                      _ptr(status), _stream(stream)),
           "gdn_prefill")


def gdn_spec_verify(dims, batch, params, qkv, a, b, o, pages, status, stream=None):
    _check(load_library().gdn_spec_verify(ctypes.byref(dims), ctypes.byref(batch),
                                          ctypes.byref(params), _ptr(qkv), _ptr(a), _ptr(b),
                                          _ptr(o), _ptr(pages), _ptr(status), _stream(stream)),
           "gdn_spec_verify")


def gdn_spec_step(dims, batch, params, x, conv_w, a, b, o, pages, status, stream=None):
    _check(load_library().gdn_spec_step(ctypes.byref(dims), ctypes.byref(batch),
                                        ctypes.byref(params), _ptr(x), _ptr(conv_w), _ptr(a),
                                        _ptr(b), _ptr(o), _ptr(pages), _ptr(status),
                                        _stream(stream)), "gdn_spec_step")


def gdn_spec_slots(dims, batch, params, x, conv_w, y, a, b, o, slots, status, stream=None):
    _check(load_library().gdn_spec_slots(ctypes.byref(dims), ctypes.byref(batch),
                                         ctypes.byref(params), _ptr(x), _ptr(conv_w), _ptr(y),
                                         _ptr(a), _ptr(b), _ptr(o), _ptr(slots), _ptr(status),
                                         _stream(stream)), "gdn_spec_slots")


def gdn_page_to_slots(dims, n, page, pool, num_pages, num_pools, pages, slots, status,
                      stream=None):
    _check(load_library().gdn_page_to_slots(ctypes.byref(dims), int(n), _ptr(page), _ptr(pool),
                                            int(num_pages), int(num_pools), _ptr(pages),
                                            _ptr(slots), _ptr(status), _stream(stream)),
           "gdn_page_to_slots")


def gdn_slots_to_page(dims, n, pool, slot, page, num_pools, num_pages, slots, pages, status,
                      stream=None):
    _check(load_library().gdn_slots_to_page(ctypes.byref(dims), int(n), _ptr(pool), _ptr(slot),
                                            _ptr(page), int(num_pools), int(num_pages),
                                            _ptr(slots), _ptr(pages), _ptr(status),
                                            _stream(stream)), "gdn_slots_to_page")


def gdn_chunk_prefill_workspace_bytes(dims, batch) -> int:
    return int(load_library().gdn_chunk_prefill_workspace_bytes(ctypes.byref(dims),
                                                                 ctypes.byref(batch)))


def gdn_chunk_prefill(dims, batch, params, qkv, a, b, o, pages, workspace, workspace_bytes,
                      status, stream=None):
    _check(load_library().gdn_chunk_prefill(ctypes.byref(dims), ctypes.byref(batch),
                                            ctypes.byref(params), _ptr(qkv), _ptr(a), _ptr(b),
                                            _ptr(o), _ptr(pages), _ptr(workspace),
                                            int(workspace_bytes), _ptr(status), _stream(stream)),
           "gdn_chunk_prefill")


def gdn_chunk_prefill_noalloc(dims, batch, params, qkv, a, b, o, pages, status, stream=None):
    _check(load_library().gdn_chunk_prefill_noalloc(ctypes.byref(dims), ctypes.byref(batch),
                                                    ctypes.byref(params), _ptr(qkv), _ptr(a),
                                                    _ptr(b), _ptr(o), _ptr(pages), _ptr(status),
                                                    _stream(stream)),
           "gdn_chunk_prefill_noalloc")


def gdn_check_bounded_wait(limit_ns, status, stream=None):
    _check(load_library().gdn_check_bounded_wait(int(limit_ns), _ptr(status), _stream(stream)),
           "gdn_check_bounded_wait")


def gdn_strerror(code: int) -> str:
    return load_library().gdn_strerror(int(code)).decode()


def gdn_abi_version() -> int:
    return int(load_library().gdn_abi_version())


def raise_on_status(status, where="device"):
    """Read the device status word (synchronises its stream) and raise if set."""
    code = int(status.item())
    if code != 0:
        raise GdnError(code, where)
