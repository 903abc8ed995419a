"""The C-ABI seen from a plain C client (no GPU needed).

A C99 program that includes only ``include/gdn.h`` is compiled with strict
warnings, linked against libgdn.so and run. It prints the size and field
offsets of every struct the header declares, the values of its enums and
flag macros, and the results of the host-only calls (layouts, strerror,
argument validation). The Python binding's ctypes view must agree with all
of it, so that a C caller and the binding describe the same boundary.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import gated_deltanet_linear_14_gb300 as gdn
from gated_deltanet_linear_14_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "gdn.h"

#define SIZE(T) printf("size %s %zu\n", #T, sizeof(T))
#define OFF(T, f) printf("off %s %s %zu\n", #T, #f, offsetof(T, f))
#define VAL(x) printf("val %s %lld\n", #x, (long long)(x))

static void dims_full(gdn_dims* d, int32_t state) {
  memset(d, 0, sizeof(*d));
  d->num_k_heads = 16; d->num_v_heads = 32; d->head_k_dim = 128;
  d->head_v_dim = 128; d->conv_width = 4; d->max_candidates = 8;
  d->io_dtype = GDN_BF16; d->state_dtype = state; d->out_dtype = GDN_BF16;
}

int main(void) {
  gdn_dims d;
  gdn_page_layout_t L;
  gdn_slot_layout_t S;
  gdn_batch b;
  gdn_params p;
  int32_t code;
  int32_t st;

  SIZE(gdn_dims); SIZE(gdn_params); SIZE(gdn_batch);
  SIZE(gdn_page_layout_t); SIZE(gdn_slot_layout_t);
  OFF(gdn_dims, num_k_heads); OFF(gdn_dims, max_candidates); OFF(gdn_dims, out_dtype);
  OFF(gdn_params, A_log); OFF(gdn_params, dt_bias); OFF(gdn_params, conv_bias);
  OFF(gdn_params, scale); OFF(gdn_params, norm_eps); OFF(gdn_params, gate_mode);
  OFF(gdn_batch, num_requests); OFF(gdn_batch, num_pages); OFF(gdn_batch, row_start);
  OFF(gdn_batch, row_len); OFF(gdn_batch, page); OFF(gdn_batch, flags);
  OFF(gdn_batch, n_accepted); OFF(gdn_batch, order);
  OFF(gdn_page_layout_t, page_bytes); OFF(gdn_page_layout_t, window_offset);
  OFF(gdn_page_layout_t, state_offset); OFF(gdn_page_layout_t, record_offset);
  OFF(gdn_page_layout_t, record_bytes); OFF(gdn_page_layout_t, flag_offset);
  OFF(gdn_slot_layout_t, pool_bytes); OFF(gdn_slot_layout_t, slot_bytes);
  OFF(gdn_slot_layout_t, state_offset); OFF(gdn_slot_layout_t, window_offset);

  VAL(GDN_F32); VAL(GDN_BF16);
  VAL(GDN_REQ_FRESH); VAL(GDN_REQ_SPEC); VAL(GDN_REQ_PARITY);
  VAL(GDN_OK); VAL(GDN_ERR_INVALID_ARG); VAL(GDN_ERR_UNSUPPORTED);
  VAL(GDN_ERR_LAUNCH); VAL(GDN_ERR_WORKSPACE); VAL(GDN_ERR_NO_DEVICE);
  VAL(GDN_DEV_BAD_PAGE); VAL(GDN_DEV_BAD_ROWS); VAL(GDN_DEV_BAD_ACCEPTED);
  VAL(GDN_DEV_STALE_STEP); VAL(GDN_DEV_TOO_MANY_CANDIDATES);
  VAL(GDN_DEV_RECORD_OPEN); VAL(GDN_DEV_BAD_FLAG); VAL(GDN_DEV_TIMEOUT);

  printf("abi %u\n", (unsigned)gdn_abi_version());

  dims_full(&d, GDN_F32);
  printf("status page_layout %d\n", (int)gdn_page_layout(&d, &L));
  printf("page %zu %zu %zu %zu %zu %zu %zu %zu\n", L.page_bytes, L.window_offset,
         L.window_bytes, L.state_offset, L.state_bytes, L.record_offset,
         L.record_bytes, L.flag_offset);
  printf("status slot_layout %d\n", (int)gdn_slot_layout(&d, &S));
  printf("slot %zu %zu %zu %zu\n", S.pool_bytes, S.slot_bytes, S.state_offset,
         S.window_offset);

  d.head_k_dim = 96;
  printf("status bad_dk %d\n", (int)gdn_page_layout(&d, &L));
  printf("status null_out %d\n", (int)gdn_page_layout(NULL, &L));

  /* host validation: a negative request count is rejected before any launch */
  dims_full(&d, GDN_F32);
  memset(&b, 0, sizeof(b));
  memset(&p, 0, sizeof(p));
  b.num_requests = -1;
  p.A_log = (const float*)&st; p.dt_bias = (const float*)&st; p.norm_eps = 1e-6f;
  code = gdn_seq(&d, &b, &p, &st, &st, &st, &st, &st, &st, NULL);
  printf("status negative_requests %d\n", (int)code);

  for (code = -5; code <= 8; ++code) printf("err %d %s\n", (int)code, gdn_strerror(code));
  return 0;
}
"""


@pytest.fixture(scope="module")
def c_client(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = gbuild.build()
    d = tmp_path_factory.mktemp("cabi")
    src = d / "client.c"
    exe = d / "client"
    src.write_text(C_SOURCE)
    libdir = os.path.dirname(lib)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-lgdn", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    out = {"size": {}, "off": {}, "val": {}, "status": {}, "err": {}}
    for line in r.stdout.splitlines():
        kind, *rest = line.split(" ")
        if kind == "size":
            out["size"][rest[0]] = int(rest[1])
        elif kind == "off":
            out["off"][(rest[0], rest[1])] = int(rest[2])
        elif kind == "val":
            out["val"][rest[0]] = int(rest[1])
        elif kind == "status":
            out["status"][rest[0]] = int(rest[1])
        elif kind == "err":
            out["err"][int(rest[0])] = " ".join(rest[1:])
        else:
            out[kind] = [int(v) for v in rest]
    return out


CTYPES = {"gdn_dims": gdn.Dims, "gdn_params": gdn.Params, "gdn_batch": gdn.Batch,
          "gdn_page_layout_t": gdn.PageLayout, "gdn_slot_layout_t": gdn.SlotLayout}


def test_struct_sizes_match_the_binding(c_client):
    for name, cls in CTYPES.items():
        assert c_client["size"][name] == ctypes.sizeof(cls), name


def test_field_offsets_match_the_binding(c_client):
    assert c_client["off"]
    for (name, field), off in c_client["off"].items():
        assert getattr(CTYPES[name], field).offset == off, (name, field)


def test_enums_and_flags_match_the_binding(c_client):
    v = c_client["val"]
    assert v["GDN_F32"] == gdn.GDN_F32 and v["GDN_BF16"] == gdn.GDN_BF16
    assert v["GDN_REQ_FRESH"] == gdn.GDN_REQ_FRESH
    assert v["GDN_REQ_SPEC"] == gdn.GDN_REQ_SPEC
    assert v["GDN_REQ_PARITY"] == gdn.GDN_REQ_PARITY
    for code, name in gdn.STATUS.items():
        assert v[name] == code, name


def test_host_calls_agree_with_the_binding(c_client):
    assert c_client["abi"] == [gdn.gdn_abi_version()]
    st = c_client["status"]
    assert st["page_layout"] == 0 and st["slot_layout"] == 0
    assert st["bad_dk"] == gdn.CODES["GDN_ERR_UNSUPPORTED"]
    assert st["null_out"] == gdn.CODES["GDN_ERR_INVALID_ARG"]
    assert st["negative_requests"] == gdn.CODES["GDN_ERR_INVALID_ARG"]
    d = gdn.make_dims(16, 32, 128, 128, 4, 8, gdn.GDN_BF16, gdn.GDN_F32, gdn.GDN_BF16)
    L = gdn.gdn_page_layout(d)
    assert c_client["page"] == [L.page_bytes, L.window_offset, L.window_bytes,
                                L.state_offset, L.state_bytes, L.record_offset,
                                L.record_bytes, L.flag_offset]
    S = gdn.gdn_slot_layout(d)
    assert c_client["slot"] == [S.pool_bytes, S.slot_bytes, S.state_offset, S.window_offset]
    for code, text in c_client["err"].items():
        assert text == gdn.gdn_strerror(code)
