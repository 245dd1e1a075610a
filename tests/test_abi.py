"""C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments on the host before any CUDA call (CPU only, no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ws_build.build()
    return ws.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ws.h")).read()
    return sorted(set(re.findall(r"WS_API\s+[\w\s\*]+?\b(ws_\w+)\s*\(", text)))


def test_header_declares_the_four_hot_path_calls():
    names = declared_symbols()
    for n in ["ws_kv_append", "ws_block_causal_attn", "ws_block_causal_prefill", "ws_fm_euler_step"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert names == sorted(ws.SIGNATURES), "binding and header disagree"
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert lib.ws_status_string(0) == b"WS_OK"
    assert lib.ws_status_string(5) == b"WS_ERR_TIMEOUT"
    assert ws.ws_abi_version() == 101


FAKE = 0x10000          # 16-byte aligned, never dereferenced by host validation


def _offs(vals):
    a = np.asarray(vals, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def test_kv_append_host_validation(lib):
    # capacity overflow
    st = lib.ws_kv_append(FAKE, FAKE, FAKE, FAKE, 10, 5, 12, 2, 128, ws.WS_BF16, None)
    assert st == ws.WS_ERR_CAPACITY and b"capacity" in lib.ws_last_error()
    # cache_len + n_new past the int64 range must not wrap into an accepted write
    big = 2 ** 63 - 1
    assert lib.ws_kv_append(FAKE, FAKE, FAKE, FAKE, big, 1, 16, 1, 128, ws.WS_BF16, None) == ws.WS_ERR_CAPACITY
    assert lib.ws_kv_append(FAKE, FAKE, FAKE, FAKE, 2 ** 62, 2 ** 62, 2 ** 62 + 5, 1, 128, ws.WS_BF16,
                            None) == ws.WS_ERR_CAPACITY
    # unknown dtype
    assert lib.ws_kv_append(FAKE, FAKE, FAKE, FAKE, 0, 1, 8, 1, 64, 7, None) == ws.WS_ERR_INVALID_ARGUMENT
    # misaligned pointer
    assert lib.ws_kv_append(FAKE + 8, FAKE, FAKE, FAKE, 0, 1, 8, 1, 64, ws.WS_BF16, None) == \
        ws.WS_ERR_INVALID_ARGUMENT
    # row not a multiple of 16 bytes
    assert lib.ws_kv_append(FAKE, FAKE, FAKE, FAKE, 0, 1, 8, 1, 4, ws.WS_BF16, None) == ws.WS_ERR_UNSUPPORTED
    # n_new == 0 is a no-op that succeeds without touching the device
    assert lib.ws_kv_append(0, 0, 0, 0, 3, 0, 8, 1, 128, ws.WS_BF16, None) == ws.WS_OK


def _attn(lib, fn, offs_vals, cap=1024, H=2, D=128, dt=ws.WS_BF16, scale=0.0, ptr=FAKE):
    arr, p = _offs(offs_vals)
    return getattr(lib, fn)(ptr, FAKE, FAKE, FAKE, None, p, FAKE, len(arr) - 1, cap, H, D,
                            scale, dt, None, 0, None)


@pytest.mark.parametrize("fn", ["ws_block_causal_attn", "ws_block_causal_prefill"])
def test_attention_host_validation(lib, fn):
    assert _attn(lib, fn, [1, 5]) == ws.WS_ERR_INVALID_ARGUMENT            # offsets[0] != 0
    assert _attn(lib, fn, [0, 5, 3]) == ws.WS_ERR_INVALID_ARGUMENT         # decreasing
    assert _attn(lib, fn, [0, 600, 1200]) == ws.WS_ERR_CAPACITY            # past capacity
    assert _attn(lib, fn, [0, 8], D=64) == ws.WS_ERR_UNSUPPORTED          # bf16 needs D=128
    assert _attn(lib, fn, [0, 8], D=96, dt=ws.WS_F32) == ws.WS_ERR_UNSUPPORTED
    assert _attn(lib, fn, [0, 8], scale=-1.0) == ws.WS_ERR_INVALID_ARGUMENT
    assert _attn(lib, fn, [0, 8], ptr=FAKE + 4) == ws.WS_ERR_INVALID_ARGUMENT
    assert _attn(lib, fn, [0, 8], ptr=0) == ws.WS_ERR_INVALID_ARGUMENT
    arr, p = _offs([0, 8])
    assert getattr(lib, fn)(FAKE, FAKE, FAKE, FAKE, None, p, FAKE, 0, 16, 1, 128, 0.0,
                            ws.WS_BF16, None, 0, None) == ws.WS_ERR_INVALID_ARGUMENT


def test_side_attention_host_validation(lib):
    f = lib.ws_block_causal_attn_side

    def call(offs_vals, ks=FAKE, vs=FAKE, dt=ws.WS_BF16, cap=1024, D=128, commit=0):
        arr, p = _offs(offs_vals)
        return f(FAKE, FAKE, FAKE, ks, vs, commit, FAKE, None, p, FAKE, len(arr) - 1, cap, 2, D, 0.0,
                 dt, None, 0, None)
    assert call([0, 8, 16], ks=0) == ws.WS_ERR_INVALID_ARGUMENT          # missing side buffer
    assert call([0, 8, 16], vs=FAKE + 8) == ws.WS_ERR_INVALID_ARGUMENT   # misaligned side buffer
    assert call([0, 8, 16], dt=ws.WS_F32) == ws.WS_ERR_UNSUPPORTED        # bf16 only
    assert call([0, 1100, 1200]) == ws.WS_ERR_CAPACITY                   # history past capacity
    assert call([0, 9, 5]) == ws.WS_ERR_INVALID_ARGUMENT                 # decreasing offsets
    assert call([0, 1000, 1100], commit=1) == ws.WS_ERR_CAPACITY          # commit needs room for the unit


def test_empty_query_block_is_a_no_op(lib):
    """An empty newest block (equal last offsets) or an empty sequence has no
    query rows: every attention call returns WS_OK before touching memory
    (the pointers here are never dereferenced)."""
    for offs_vals in ([0, 8, 8], [0, 0], [0, 0, 0]):
        arr, p = _offs(offs_vals)
        for fn in ("ws_block_causal_attn", "ws_block_causal_prefill"):
            if fn == "ws_block_causal_prefill" and offs_vals[-1] != 0:
                continue                      # the prefill has rows there
            assert getattr(lib, fn)(FAKE, FAKE, FAKE, FAKE, None, p, FAKE, len(arr) - 1, 64, 2, 128,
                                    0.0, ws.WS_BF16, None, 0, None) == ws.WS_OK
        assert lib.ws_block_causal_attn_side(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, None, p, FAKE,
                                             len(arr) - 1, 64, 2, 128, 0.0, ws.WS_BF16, None, 0,
                                             None) == ws.WS_OK


def test_euler_host_validation(lib):
    assert lib.ws_fm_euler_step(FAKE, ws.WS_BF16, FAKE, ws.WS_BF16, None, 8, 0.25, None) == ws.WS_ERR_UNSUPPORTED
    assert lib.ws_fm_euler_step(FAKE, ws.WS_F32, FAKE + 4, ws.WS_BF16, None, 8, 0.25, None) == \
        ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_fm_euler_step(FAKE, ws.WS_F32, FAKE, ws.WS_BF16, None, 8, float("inf"), None) == \
        ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_fm_euler_step(0, ws.WS_F32, 0, ws.WS_BF16, None, 0, 0.25, None) == ws.WS_OK


def test_euler_cfg_host_validation(lib):
    f = lib.ws_fm_euler_cfg_step
    assert f(FAKE, ws.WS_BF16, FAKE, FAKE, ws.WS_BF16, None, 8, 2.0, 0.25, None) == ws.WS_ERR_UNSUPPORTED
    assert f(FAKE, ws.WS_F32, FAKE, FAKE + 4, ws.WS_BF16, None, 8, 2.0, 0.25, None) == ws.WS_ERR_INVALID_ARGUMENT
    assert f(FAKE, ws.WS_F32, FAKE, FAKE, ws.WS_BF16, None, 8, float("nan"), 0.25, None) == \
        ws.WS_ERR_INVALID_ARGUMENT
    assert f(FAKE, ws.WS_F32, 0, FAKE, ws.WS_BF16, None, 8, 2.0, 0.25, None) == ws.WS_ERR_INVALID_ARGUMENT
    assert f(0, ws.WS_F32, 0, 0, ws.WS_BF16, None, 0, 2.0, 0.25, None) == ws.WS_OK


def test_timeout_setting_rejects_zero(lib):
    assert lib.ws_set_wait_timeout_ns(0) == ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_set_wait_timeout_ns(2_000_000_000) == ws.WS_OK


def test_binding_raises_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ws, "_lib", None)
    monkeypatch.setattr(ws, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ws.load()


def _header_params():
    """{function name: parameter count} from the WS_API declarations."""
    text = open(os.path.join(ROOT, "include", "ws.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"WS_API\s+[\w\s\*]+?\b(ws_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = len(params)
    return out


def test_binding_argument_counts_match_the_header():
    params = _header_params()
    assert set(params) == set(ws.SIGNATURES)
    for name, (_, argtypes) in ws.SIGNATURES.items():
        assert len(argtypes) == params[name], name


def test_header_is_plain_c_and_links(lib, tmp_path):
    """A C99 translation unit that includes ws.h and calls every entry point
    compiles without warnings and links against the built library (it is not
    run: no GPU is needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_ws.c"
    src.write_text(r'''
#include <stdio.h>
#include "ws.h"
int main(void) {
  int32_t offs[3] = {0, 8, 16};
  int code = 0, info = 0;
  ws_stream_t s = NULL;
  ws_status st = ws_kv_append(NULL, NULL, NULL, NULL, 0, 0, 16, 1, 128, WS_BF16, s);
  st |= ws_block_causal_attn(NULL, NULL, NULL, NULL, NULL, offs, NULL, 2, 16, 1, 128, 0.f, WS_BF16, NULL, 0, s);
  st |= ws_block_causal_attn_side(NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL, offs, NULL, 2, 16, 1, 128, 0.f,
                                  WS_BF16, NULL, 0, s);
  st |= ws_block_causal_attn_noalloc(NULL, NULL, NULL, NULL, NULL, offs, NULL, 2, 16, 1, 128, 0.f, WS_BF16, s);
  st |= ws_block_causal_prefill(NULL, NULL, NULL, NULL, NULL, offs, NULL, 2, 16, 1, 128, 0.f, WS_BF16, NULL, 0, s);
  st |= ws_fm_euler_step(NULL, WS_F32, NULL, WS_BF16, NULL, 0, 0.25f, s);
  st |= ws_fm_euler_cfg_step(NULL, WS_F32, NULL, NULL, WS_BF16, NULL, 0, 2.f, 0.25f, s);
  size_t n = ws_block_causal_attn_workspace_size(8, 16, 1, 128);
  st |= ws_get_device_error(&code, &info);
  st |= ws_clear_device_error();
  st |= ws_set_wait_timeout_ns(1000000000ull);
  st |= ws_debug_force_wait_timeout(0);
  printf("%s %s %zu %d\n", ws_status_string(st), ws_last_error(), n, ws_abi_version());
  return 0;
}
''')
    lib_dir = os.path.dirname(ws_build.LIB_PATH)
    res = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                          str(src), "-L", lib_dir, "-l:" + os.path.basename(ws_build.LIB_PATH),
                          "-o", str(tmp_path / "use_ws")], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_binding_rejects_shapes_the_abi_cannot_see():
    """The C ABI takes pointers only; the binding checks what they must hold
    (a wrong row count or a smaller V cache would be read past its end)."""
    import torch
    H, D = 2, 128
    bf = torch.bfloat16
    k = torch.zeros(H, 64, D, dtype=bf)
    offs = [0, 40, 60]
    offs_dev = torch.tensor(offs, dtype=torch.int32)
    q = torch.zeros(20, H, D, dtype=bf)
    out = torch.empty_like(q)
    with pytest.raises(ValueError, match="v_cache"):
        ws.ws_block_causal_attn(q, k, torch.zeros(H, 32, D, dtype=bf), out, offs, offs_dev)
    with pytest.raises(ValueError, match="rows"):
        ws.ws_block_causal_attn(q[:10], k, k, out[:10], offs, offs_dev)
    with pytest.raises(ValueError, match="rows"):
        ws.ws_block_causal_attn_noalloc(q[:19], k, k, out[:19], offs, offs_dev)
    with pytest.raises(ValueError, match="rows"):
        ws.ws_block_causal_attn_side(q[:5], k, k, q[:5], q[:5], out[:5], offs, offs_dev)
    with pytest.raises(ValueError, match="rows"):          # prefill reads all 60 tokens
        ws.ws_block_causal_prefill(q, k, k, out, offs, offs_dev)
    # consistent shapes get past the shape checks (and stop at the device check here)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ws.ws_block_causal_attn(q, k, k, out, offs, offs_dev)
    full = torch.zeros(60, H, D, dtype=bf)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ws.ws_block_causal_prefill(full, k, k, torch.empty_like(full), offs, offs_dev)


def test_device_resident_entry_points_host_validation(lib):
    """The device-resident-size variants check on the host everything that
    does not depend on the sizes the kernels read at run time."""
    # append: n_max above capacity, unsupported row size, null state, misaligned state
    assert lib.ws_kv_append_dev(FAKE, FAKE, FAKE, FAKE, FAKE, 20, 10, 2, 128, ws.WS_BF16, None) \
        == ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_kv_append_dev(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 2, 4, ws.WS_BF16, None) \
        == ws.WS_ERR_UNSUPPORTED
    assert lib.ws_kv_append_dev(FAKE, FAKE, FAKE, FAKE, None, 4, 10, 2, 128, ws.WS_BF16, None) \
        == ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_kv_append_dev(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 4, 10, 2, 128, ws.WS_BF16, None) \
        == ws.WS_ERR_INVALID_ARGUMENT
    # attention: only bf16 with head_dim 128; q_max within capacity; workspace required
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, st=FAKE, q_max=300, cap=1000, h=2, d=128,
                scale=0.0, dt=ws.WS_BF16, wsp=FAKE, wsb=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return lib.ws_block_causal_attn_dev(a["q"], a["k"], a["v"], a["o"], a["lse"], a["st"], a["q_max"],
                                            a["cap"], a["h"], a["d"], a["scale"], a["dt"], a["wsp"],
                                            a["wsb"], None)
    assert call(dt=ws.WS_F32) == ws.WS_ERR_UNSUPPORTED
    assert call(d=64) == ws.WS_ERR_UNSUPPORTED
    assert call(q_max=2000) == ws.WS_ERR_INVALID_ARGUMENT
    assert call(q_max=0) == ws.WS_ERR_INVALID_ARGUMENT
    assert call(wsp=None) == ws.WS_ERR_INVALID_ARGUMENT
    assert call(st=None) == ws.WS_ERR_INVALID_ARGUMENT
    assert call(scale=-1.0) == ws.WS_ERR_INVALID_ARGUMENT
    assert call(q=FAKE + 8) == ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_block_causal_attn_dev_workspace_size(0, 10, 2, 128) == ctypes.c_size_t(-1).value
    assert lib.ws_block_causal_attn_dev_workspace_size(20, 10, 2, 128) == ctypes.c_size_t(-1).value
    # state advance: null state, negative size count
    assert lib.ws_unit_state_advance(None, FAKE, 3, None) == ws.WS_ERR_INVALID_ARGUMENT
    assert lib.ws_unit_state_advance(FAKE, FAKE, -1, None) == ws.WS_ERR_INVALID_ARGUMENT
