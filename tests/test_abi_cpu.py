"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol the header declares, the ctypes mirror matches the C struct layout,
and host-side validation rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import masked_gqa_attention_gb300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "masked_gqa_attn.h")


@pytest.fixture(scope="module")
def L():
    M.build_library()
    return M.lib()


DEBUG_HEADER = os.path.join(ROOT, "include", "masked_gqa_attn_debug.h")


def declared_symbols(header=HEADER):
    text = open(header).read()
    return re.findall(r"MGQA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    assert set(syms) == set(M.EXPORTED_SYMBOLS), syms


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
    assert L.mgqa_abi_version() == 6
    assert L.mgqa_status_string(M.MGQA_ERR_TIMEOUT) == b"device wait timed out"
    assert b"debug" in L.mgqa_status_string(M.MGQA_ERR_DEVICE_CHECK)


def test_debug_library_exports_the_debug_entry_points(L):
    assert set(declared_symbols(DEBUG_HEADER)) == set(M.DEBUG_SYMBOLS)
    Ld = M.debug_lib()
    for name in declared_symbols() + declared_symbols(DEBUG_HEADER):
        assert hasattr(Ld, name), name
    # the product library carries none of the test equipment
    for name in M.DEBUG_SYMBOLS:
        assert not hasattr(L, name), name


def test_debug_counter_count_is_checked_on_the_host(L):
    Ld = M.debug_lib()
    buf = (ctypes.c_uint64 * 8)()
    assert Ld.mgqa_debug_counters(buf, 8) == M.MGQA_ERR_INVALID_ARG
    assert Ld.mgqa_debug_inject_prefill_stall(0, 1000) == M.MGQA_ERR_INVALID_ARG


@pytest.mark.parametrize("cname,py", [("mgqa_args", M.MgqaArgs), ("mgqa_rope_args", M.MgqaRopeArgs),
                                     ("mgqa_qk_rope", M.MgqaQkRope)])
def test_struct_layout_matches_header(tmp_path, cname, py):
    fields = [f for f, _ in py._fields_]
    src = tmp_path / "off.c"
    body = "\n".join(f'printf("{f} %zu\\n", offsetof({cname}, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "masked_gqa_attn.h"\n'
                   f'int main(void){{ {body} printf("size %zu\\n", sizeof({cname})); return 0; }}\n')
    exe = tmp_path / "off"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.split() for line in out if line)
    for f in fields:
        assert int(got[f]) == getattr(py, f).offset, f
    assert int(got["size"]) == ctypes.sizeof(py)


def _valid_args():
    a = M.MgqaArgs()
    a.dtype = M.MGQA_BF16
    a.B, a.Hq, a.Hkv, a.Lq, a.Lk, a.D = 2, 16, 8, 1024, 1024, 128
    base = 1 << 20  # fake, never dereferenced: validation fails before any launch
    a.q, a.k, a.v, a.out = base, base * 2, base * 3, base * 4
    for fld, H in (("q_stride", 16), ("k_stride", 8), ("v_stride", 8), ("o_stride", 16)):
        getattr(a, fld)[:] = [H * 1024 * 128, 1024 * 128, 128]
    a.scale = 0.088
    return a


@pytest.mark.parametrize("mutate,code", [
    (lambda a: setattr(a, "Hkv", 3), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "D", 96), M.MGQA_ERR_UNSUPPORTED),
    (lambda a: setattr(a, "B", 0), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "Lk", 0), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "q", 0), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "k", (1 << 20) + 8), M.MGQA_ERR_INVALID_ARG),
    (lambda a: a.k_stride.__setitem__(2, 100), M.MGQA_ERR_INVALID_ARG),
    (lambda a: a.v_stride.__setitem__(1, -128), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "scale", float("nan")), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "scale", float("inf")), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "dtype", 7), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "seg_q", 1 << 22), M.MGQA_ERR_INVALID_ARG),
    (lambda a: (setattr(a, "mask_bits", 1 << 22), setattr(a, "mask_stride_q", 8)), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "mask_bits", (1 << 22) + 2), M.MGQA_ERR_INVALID_ARG),
    (lambda a: setattr(a, "lse", (1 << 22) + 1), M.MGQA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_arguments(L, mutate, code):
    a = _valid_args()
    mutate(a)
    st = L.masked_gqa_attn_prefill(ctypes.byref(a), None)
    assert st == code, L.mgqa_last_error_detail()
    assert L.mgqa_last_error_detail() != b""


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="on a GPU machine the call would launch on the fake pointers")
@pytest.mark.parametrize("sq,sb", [(0, 32), (0, 0), (32, 0)])
def test_broadcast_mask_strides_pass_validation(L, sq, sb):
    # one key-padding row per batch row ([B][1][W], query stride 0) or one
    # mask for the whole batch (batch stride 0): validation accepts both, so
    # without a GPU the call fails only later, at the launch
    a = _valid_args()
    a.mask_bits = 1 << 22
    a.mask_stride_q, a.mask_stride_b = sq, sb
    st = L.masked_gqa_attn_prefill(ctypes.byref(a), None)
    assert st == M.MGQA_ERR_CUDA, L.mgqa_last_error_detail()


def test_null_args_rejected(L):
    assert L.masked_gqa_attn_prefill(None, None) == M.MGQA_ERR_INVALID_ARG
    assert L.masked_gqa_attn_decode(None, None, 0, None) == M.MGQA_ERR_INVALID_ARG
    assert L.masked_gqa_attn_decode_workspace_size(None) == 0


def test_decode_validation(L):
    a = _valid_args()
    assert L.masked_gqa_attn_decode_workspace_size(ctypes.byref(a)) == 0  # Lq != 1
    assert L.masked_gqa_attn_decode(ctypes.byref(a), None, 0, None) == M.MGQA_ERR_INVALID_ARG
    a.Lq = 1
    a.B, a.Hq, a.Hkv, a.Lk, a.D = 8, 16, 2, 8192, 64
    # merged on chip: a nominal, shape-independent size (non-zero = valid)
    assert L.masked_gqa_attn_decode_workspace_size(ctypes.byref(a)) == 16
    a.B, a.Hq = 4096, 64
    assert L.masked_gqa_attn_decode_workspace_size(ctypes.byref(a)) == 16
    a.Lk = 32769  # past the longest cache the chunk masks cover
    assert L.masked_gqa_attn_decode_workspace_size(ctypes.byref(a)) == 0
    assert L.masked_gqa_attn_decode_static(ctypes.byref(a), None) == M.MGQA_ERR_UNSUPPORTED


def test_decode_ignores_the_workspace_arguments(L):
    # valid arguments get past validation with or without a workspace, so
    # without a GPU the call fails only at the launch
    a = _valid_args()
    a.Lq, a.B, a.Hq, a.Hkv, a.Lk, a.D = 1, 8, 16, 2, 8192, 64
    for ws, n in ((None, 0), (1 << 20, 16), ((1 << 20) + 4, 3)):
        assert L.masked_gqa_attn_decode(ctypes.byref(a), ws, n, None) == M.MGQA_ERR_CUDA
    assert L.masked_gqa_attn_decode_static(ctypes.byref(a), None) == M.MGQA_ERR_CUDA


def _valid_rope():
    a = M.MgqaRopeArgs()
    a.dtype = M.MGQA_BF16
    a.B, a.H, a.L, a.D = 2, 16, 1024, 128
    a.x = 1 << 20  # fake, never dereferenced: validation fails before any launch
    a.x_stride[:] = [16 * 1024 * 128, 1024 * 128, 128]
    a.inv_freq = 1 << 22
    a.rot_dim, a.heads, a.interleaved = 64, 1, 1
    return a


@pytest.mark.parametrize("mutate", [
    lambda a: setattr(a, "rot_dim", 63),
    lambda a: setattr(a, "rot_dim", 0),
    lambda a: setattr(a, "rot_dim", 130),
    lambda a: setattr(a, "heads", 0),
    lambda a: setattr(a, "heads", 17),
    lambda a: setattr(a, "L", 0),
    lambda a: setattr(a, "dtype", 5),
    lambda a: setattr(a, "x", 0),
    lambda a: setattr(a, "inv_freq", 0),
    lambda a: setattr(a, "x", (1 << 20) + 1),
    lambda a: setattr(a, "inv_freq", (1 << 22) + 2),
    lambda a: setattr(a, "positions", (1 << 23) + 2),
    lambda a: a.x_stride.__setitem__(1, -1),
    lambda a: a.x_stride.__setitem__(2, 0),  # rows would share elements
])
def test_rope_rejects_bad_arguments(L, mutate):
    a = _valid_rope()
    mutate(a)
    assert L.masked_gqa_rope(ctypes.byref(a), None) == M.MGQA_ERR_INVALID_ARG
    assert L.mgqa_last_error_detail() != b""
    assert L.masked_gqa_rope(None, None) == M.MGQA_ERR_INVALID_ARG
    # the pair entry checks both tensors before anything is enqueued and names the bad one
    good = _valid_rope()
    good.x = 1 << 24
    assert L.masked_gqa_rope_pair(ctypes.byref(a), ctypes.byref(good), None) == M.MGQA_ERR_INVALID_ARG
    assert b"(q)" in L.mgqa_last_error_detail()
    assert L.masked_gqa_rope_pair(ctypes.byref(good), ctypes.byref(a), None) == M.MGQA_ERR_INVALID_ARG
    assert b"(k)" in L.mgqa_last_error_detail()


def test_rope_pair_rejects_mixed_dtypes_and_null(L):
    q, k = _valid_rope(), _valid_rope()
    k.x = 1 << 24
    k.dtype = M.MGQA_FP16
    assert L.masked_gqa_rope_pair(ctypes.byref(q), ctypes.byref(k), None) == M.MGQA_ERR_INVALID_ARG
    assert b"dtypes differ" in L.mgqa_last_error_detail()
    assert L.masked_gqa_rope_pair(ctypes.byref(q), None, None) == M.MGQA_ERR_INVALID_ARG
    assert L.masked_gqa_rope_pair(None, ctypes.byref(q), None) == M.MGQA_ERR_INVALID_ARG


def test_plain_c_program_links_and_calls_the_library(L, tmp_path):
    # the boundary is a C ABI: a C program that includes only the header links
    # libmgqa.so and gets the documented status codes (no GPU needed for these)
    src = tmp_path / "use.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "masked_gqa_attn.h"
int main(void) {
  if (mgqa_abi_version() != MGQA_ABI_VERSION) return 1;
  if (masked_gqa_attn_prefill(NULL, NULL) != MGQA_ERR_INVALID_ARG) return 2;
  if (strlen(mgqa_last_error_detail()) == 0) return 3;
  mgqa_args a;
  memset(&a, 0, sizeof a);
  a.dtype = MGQA_BF16; a.B = 1; a.Hq = 4; a.Hkv = 3; a.Lq = 8; a.Lk = 8; a.D = 64;
  if (masked_gqa_attn_prefill(&a, NULL) != MGQA_ERR_INVALID_ARG) return 4;  /* Hq % Hkv */
  if (masked_gqa_attn_decode_workspace_size(&a) != 0) return 5;
  mgqa_rope_args r;
  memset(&r, 0, sizeof r);
  if (masked_gqa_rope(&r, NULL) != MGQA_ERR_INVALID_ARG) return 6;
  printf("%s\n", mgqa_status_string(MGQA_ERR_UNSUPPORTED));
  return 0;
}
''')
    exe = tmp_path / "use"
    libdir = os.path.dirname(M._LIB_PATH)
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), "-I", "/usr/local/cuda/include", str(src),
                    "-L", libdir, "-lmgqa", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() != ""


def _valid_qk_rope():
    r = M.MgqaQkRope()
    r.inv_freq = 1 << 22  # fake, never dereferenced: validation fails before any launch
    r.rot_dim, r.interleaved, r.q_heads, r.k_heads = 128, 0, 16, 8
    r.norm_eps = 1e-6
    return r


@pytest.mark.parametrize("mutate", [
    lambda r: setattr(r, "inv_freq", 0),
    lambda r: setattr(r, "inv_freq", (1 << 22) + 2),
    lambda r: setattr(r, "rot_dim", 127),
    lambda r: setattr(r, "rot_dim", 130),
    lambda r: setattr(r, "q_heads", 0),
    lambda r: setattr(r, "q_heads", 17),
    lambda r: setattr(r, "positions", (1 << 23) + 1),
    lambda r: (setattr(r, "q_norm_weight", 1 << 23), setattr(r, "norm_eps", -1.0)),
    lambda r: (setattr(r, "q_norm_weight", 1 << 23), setattr(r, "norm_eps", float("nan"))),
    lambda r: setattr(r, "k_norm_weight", (1 << 23) + 2),
])
def test_fused_rope_arguments_are_checked(L, mutate):
    r = _valid_qk_rope()
    mutate(r)
    a = _valid_args()
    assert L.masked_gqa_attn_prefill_rope(ctypes.byref(a), ctypes.byref(r), None) == M.MGQA_ERR_INVALID_ARG
    assert L.mgqa_last_error_detail() != b""


def test_fused_rope_decode_arguments_are_checked(L):
    a = _valid_args()
    a.Lq, a.Hkv = 1, 8
    a.kv_len = 1 << 22
    r = _valid_qk_rope()
    r.k_heads = 9  # more than Hkv
    st = L.masked_gqa_attn_decode_append_rope(ctypes.byref(a), 1 << 20, 1 << 20,
                                              (ctypes.c_int64 * 2)(1024, 128), (ctypes.c_int64 * 2)(1024, 128),
                                              None, ctypes.byref(r), 1 << 20, 1 << 20, None)
    assert st == M.MGQA_ERR_INVALID_ARG and b"k_heads" in L.mgqa_last_error_detail()
    assert L.masked_gqa_attn_prefill_rope(ctypes.byref(a), None, None) == M.MGQA_ERR_INVALID_ARG


def test_fused_rope_prefill_refuses_fp32(L):
    a = _valid_args()
    a.dtype = M.MGQA_FP32
    for fld, H in (("q_stride", 16), ("k_stride", 8), ("v_stride", 8), ("o_stride", 16)):
        getattr(a, fld)[:] = [H * 1024 * 128, 1024 * 128, 128]
    r = _valid_qk_rope()
    assert L.masked_gqa_attn_prefill_rope(ctypes.byref(a), ctypes.byref(r), None) == M.MGQA_ERR_UNSUPPORTED
