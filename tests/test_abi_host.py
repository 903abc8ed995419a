"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, computes layouts, and rejects bad arguments before launching
anything."""
import ctypes
import os
import re

import pytest

import gated_deltanet_linear_14_gb300 as gdn
from gated_deltanet_linear_14_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load_library()


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["gdn_conv", "gdn_seq", "gdn_spec_verify", "gdn_chunk_prefill",
              "gdn_page_layout", "gdn_strerror"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_abi_version(lib):
    assert gdn.gdn_abi_version() >> 16 == 2


def full_dims(Kc=8, state=gdn.GDN_F32, io=gdn.GDN_BF16):
    return gdn.make_dims(16, 32, 128, 128, 4, Kc, io, state, gdn.GDN_BF16)


def test_page_layout_full_shapes(lib):
    L = gdn.gdn_page_layout(full_dims())
    assert L.state_bytes == 32 * 128 * 128 * 4            # 2 MiB fp32 state
    assert L.window_bytes == (3 + 8) * 8192 * 2
    rec_row = (8192 + 64)                                  # already 16-byte aligned in bf16
    # both slots' rows, per slot and value head 216 fp32 run coefficients, and
    # per value head and candidate the fp32 u of every value column
    assert L.record_bytes == 2 * 8 * rec_row * 2 + 2 * 32 * 216 * 4 + 32 * 8 * 128 * 4
    for off in (L.state_offset, L.window_offset, L.record_offset, L.flag_offset, L.page_bytes):
        assert off % 256 == 0
    assert L.window_offset >= L.state_offset + L.state_bytes
    assert L.record_offset >= L.window_offset + L.window_bytes
    assert L.flag_offset >= L.record_offset + L.record_bytes
    assert L.page_bytes >= L.flag_offset + 4
    Lb = gdn.gdn_page_layout(full_dims(state=gdn.GDN_BF16))
    assert Lb.state_bytes == L.state_bytes // 2


def test_record_rows_padded_to_16_bytes(lib):
    # Hv = 2 with fp32 io: C + 2*Hv = 196 floats = 784 bytes (already aligned);
    # Hv = 1, Hk = 1, Dk = 32: C = 96, + 2 = 98 floats -> padded to 100
    d = gdn.make_dims(1, 1, 32, 32, 4, 8, gdn.GDN_F32, gdn.GDN_F32, gdn.GDN_F32)
    L = gdn.gdn_page_layout(d)
    assert L.record_bytes == 2 * 8 * 100 * 4 + 2 * 1 * 216 * 4 + 1 * 8 * 32 * 4


def test_slot_layout(lib):
    S = gdn.gdn_slot_layout(full_dims())
    assert S.slot_bytes % 256 == 0 and S.window_offset % 256 == 0
    assert S.window_offset >= 32 * 128 * 128 * 4
    assert S.pool_bytes == 8 * S.slot_bytes


@pytest.mark.parametrize("field,value,code", [
    ("head_k_dim", 96, -2), ("head_v_dim", 64, -2), ("conv_width", 3, -2),
    ("max_candidates", 9, -2), ("num_k_heads", 3, -2), ("num_v_heads", 0, -1),
    ("io_dtype", 5, -1), ("state_dtype", -1, -1), ("max_candidates", -1, -1),
])
def test_bad_dims_rejected(lib, field, value, code):
    d = full_dims()
    setattr(d, field, value)
    L = gdn.PageLayout()
    assert lib.gdn_page_layout(ctypes.byref(d), ctypes.byref(L)) == code


def _call_all(lib, dims, batch, params, ptr=1):
    """Call every compute entry with fake non-null pointers; all must fail on
    the host (these arguments never reach a launch)."""
    D, B, P = ctypes.byref(dims), ctypes.byref(batch), ctypes.byref(params)
    return [
        lib.gdn_conv(D, B, P, ptr, ptr, ptr, 1, ptr, ptr, None),
        lib.gdn_seq(D, B, P, ptr, ptr, ptr, ptr, ptr, ptr, None),
        lib.gdn_spec_verify(D, B, P, ptr, ptr, ptr, ptr, ptr, ptr, None),
        lib.gdn_spec_slots(D, B, P, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, None),
        lib.gdn_chunk_prefill(D, B, P, ptr, ptr, ptr, ptr, ptr, ptr, 1 << 30, ptr, None),
    ]


def _batch(R=4, rows=4, ptr=8):
    return gdn.make_batch(R, rows, 1, R, ptr, ptr, ptr, ptr, ptr, None)


def test_host_validation_rejects_before_launch(lib):
    params = gdn.make_params(8, 8)
    # negative counts
    assert set(_call_all(lib, full_dims(), _batch(R=-1), params)) == {-1}
    # too many requests for the grid
    assert set(_call_all(lib, full_dims(), _batch(R=70000), params)) == {-2}
    # missing row-map arrays
    b = _batch()
    b.row_len = None
    assert set(_call_all(lib, full_dims(), b, params)) == {-1}
    # bad gate mode / eps
    p = gdn.make_params(8, 8, gate_mode=2)
    assert set(_call_all(lib, full_dims(), _batch(), p)) == {-1}
    p = gdn.make_params(8, 8, norm_eps=-1.0)
    assert set(_call_all(lib, full_dims(), _batch(), p)) == {-1}
    # unsupported dims
    d = full_dims()
    d.head_k_dim = 256
    assert set(_call_all(lib, d, _batch(), params)) == {-2}


def test_verify_needs_a_record_and_accepted_counts(lib):
    params = gdn.make_params(8, 8)
    D0 = full_dims(Kc=0)
    b = _batch()
    assert lib.gdn_spec_verify(ctypes.byref(D0), ctypes.byref(b), ctypes.byref(params),
                               8, 8, 8, 8, 8, 8, None) == -2
    b.n_accepted = None
    D = full_dims()
    assert lib.gdn_spec_verify(ctypes.byref(D), ctypes.byref(b), ctypes.byref(params),
                               8, 8, 8, 8, 8, 8, None) == -1


def test_null_buffers_rejected(lib):
    params = gdn.make_params(8, 8)
    D, B, P = ctypes.byref(full_dims()), ctypes.byref(_batch()), ctypes.byref(params)
    assert lib.gdn_seq(D, B, P, None, 8, 8, 8, 8, 8, None) == -1       # qkv
    assert lib.gdn_seq(D, B, P, 8, 8, 8, 8, None, 8, None) == -1       # pages
    assert lib.gdn_seq(D, B, P, 8, 8, 8, 8, 8, None, None) == -1       # status
    assert lib.gdn_conv(D, B, P, 8, None, 8, 1, 8, 8, None) == -1      # conv_w
    assert lib.gdn_conv(D, B, P, 8, 8, 8, 7, 8, 8, None) == -1         # y dtype
    p2 = gdn.make_params(None, 8)
    assert lib.gdn_seq(D, B, ctypes.byref(p2), 8, 8, 8, 8, 8, 8, None) == -1


def test_empty_batch_is_a_no_op(lib):
    params = gdn.make_params(8, 8)
    b = gdn.make_batch(0, 0, 0, 0, None, None, None, None, None, None)
    D, B, P = ctypes.byref(full_dims()), ctypes.byref(b), ctypes.byref(params)
    assert lib.gdn_seq(D, B, P, None, None, None, None, None, None, None) == 0
    assert lib.gdn_conv(D, B, P, None, None, None, 1, None, None, None) == 0


def test_strerror_covers_every_code(lib):
    for code in gdn.STATUS:
        assert gdn.gdn_strerror(code) != "unknown status"
    assert gdn.gdn_strerror(12345) == "unknown status"


def test_bounded_wait_check_validates_arguments(lib):
    assert lib.gdn_check_bounded_wait(1000, None, None) == -1          # no status word
    assert lib.gdn_check_bounded_wait(0, 8, None) == -1                 # limit <= 0
    assert lib.gdn_check_bounded_wait(-5, 8, None) == -1
    assert lib.gdn_check_bounded_wait(10 ** 10 + 1, 8, None) == -1      # above 10 s


def _widest_group(lib, entry, io, state):
    """Largest number of value heads per q/k head (Dk = Dv = 128) that the
    entry accepts: the shared-memory fit is checked on the host before any
    launch (an empty batch then returns GDN_OK)."""
    params = gdn.make_params(8, 8)
    b = _batch(R=0, rows=0)
    widest = 0
    for gh in range(1, 200):
        d = gdn.make_dims(1, gh, 128, 128, 4, 8, io, state, gdn.GDN_BF16)
        D, B, P = ctypes.byref(d), ctypes.byref(b), ctypes.byref(params)
        if entry == "verify":
            rc = lib.gdn_spec_verify(D, B, P, 8, 8, 8, 8, 8, 8, None)
        elif entry == "step":
            rc = lib.gdn_spec_step(D, B, P, 8, 8, 8, 8, 8, 8, 8, None)
        else:
            rc = lib.gdn_spec_slots(D, B, P, 8, 8, 8, 8, 8, 8, 8, 8, None)
        if rc != 0:
            assert rc == gdn.CODES["GDN_ERR_UNSUPPORTED"], (entry, gh, rc)
            break
        widest = gh
    return widest


def test_each_spec_entry_checks_only_its_own_kernels(lib):
    """gdn_spec_verify is limited only by its coefficient and item kernels,
    not by the wider shared-memory needs of the one-launch step (which stages
    the group's rows and u) or of the slot kernel (the group's rows). The
    figures are the ones include/gdn.h quotes."""
    bf, f32 = gdn.GDN_BF16, gdn.GDN_F32
    assert _widest_group(lib, "verify", bf, f32) == 124
    assert _widest_group(lib, "step", bf, f32) == 18
    assert _widest_group(lib, "slots", bf, f32) == 42
