"""The C-ABI library loads and exports what include/dv.h declares (no GPU).

No test here launches a kernel: only host-side entry points (sizes, status
strings) and argument checks that fail before any CUDA call are exercised.
"""

import ctypes as C
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dv.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dv_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


def test_every_declared_symbol_is_exported(dv):
    names = _declared_functions()
    assert len(names) >= 12
    lib = C.CDLL(dv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dv.EXPORTED)


def test_struct_layouts_match_header(dv, tmp_path):
    src = tmp_path / "sizes.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "dv.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(dv_layer_desc),"
        " offsetof(dv_layer_desc, ln_eps), offsetof(dv_layer_desc, kv_cap),"
        " sizeof(dv_layer_weights), sizeof(dv_selection));return 0;}\n")
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got == [C.sizeof(dv.LayerDesc), dv.LayerDesc.ln_eps.offset, dv.LayerDesc.kv_cap.offset,
                   C.sizeof(dv.LayerWeights), C.sizeof(dv.Selection)]


def test_status_strings_and_version(dv):
    assert dv.abi_version() == 2
    for s in range(0, 8):
        assert len(dv.status_string(s)) > 0
    assert dv.status_string(0) == "ok"


def test_workspace_size_validates_desc(dv):
    good = dv.make_desc(12288, 96, 128, 49152, 1000, dv.DV_F16, 2049)
    n1 = dv.workspace_size(good, 1)
    n8 = dv.workspace_size(good, 8)
    assert 0 < n1 < n8 < (1 << 32)
    assert dv.workspace_size(good, 0) == 0
    assert dv.workspace_size(good, dv.DV_MAX_BATCH + 1) == 0
    assert dv.workspace_size(dv.make_desc(12288, 96, 96, 49152, 1000, dv.DV_F16, 2049), 1) == 0
    assert dv.workspace_size(dv.make_desc(12290, 96, 128, 49152, 1000, dv.DV_F16, 2049), 1) == 0
    assert dv.workspace_size(dv.make_desc(256, 8, 32, 1024, 32, 7, 65), 1) == 0
    assert dv.workspace_size(dv.make_desc(256, 8, 32, 1024, 32, dv.DV_F32, 0), 1) == 0
    assert dv.workspace_size(dv.make_desc(256, 8, 32, 1024, 32, dv.DV_F32, 65, ln_eps=0.0), 1) == 0
    assert dv.dv_layer_decode_launches(good, 1) == 7
    assert dv.dv_layer_decode_launches(good, 3) == 7
    assert dv.dv_layer_decode_launches(good, 0) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake-pointer checks run only without a GPU")
def test_argument_checks_fail_before_any_launch(dv):
    lib = dv._lib
    desc = dv.make_desc(256, 8, 32, 1024, 32, dv.DV_F32, 65)
    fake = [C.c_void_p(0x100000 + 256 * i) for i in range(16)]
    w = dv.LayerWeights(*fake[:15])
    sel = dv.Selection(*fake[:6])
    ws = C.c_void_p(0x200000)
    # null weights
    assert lib.dv_layer_decode(C.byref(desc), None, fake[0], None, 1, 2, 103, fake[1], fake[2], 64,
                               C.byref(sel), None, fake[3], ws, 1 << 30, None) == dv.DV_ERR_INVALID_ARG
    bad = [
        dict(batch=0), dict(batch=33), dict(kh=0), dict(kh=9), dict(kn=0), dict(kn=1025),
        dict(kv_len=-1), dict(kv_len=65),
    ]
    for b in bad:
        a = dict(batch=1, kh=2, kn=103, kv_len=64)
        a.update(b)
        assert lib.dv_layer_decode(C.byref(desc), C.byref(w), fake[0], None, a["batch"], a["kh"],
                                   a["kn"], fake[1], fake[2], a["kv_len"], C.byref(sel), None,
                                   fake[3], ws, 1 << 30, None) == dv.DV_ERR_INVALID_ARG, b
    # misaligned activation pointer
    assert lib.dv_layer_decode(C.byref(desc), C.byref(w), C.c_void_p(0x100004), None, 1, 2, 103,
                               fake[1], fake[2], 64, C.byref(sel), None, fake[3], ws, 1 << 30,
                               None) == dv.DV_ERR_INVALID_ARG
    # workspace too small / misaligned
    assert lib.dv_layer_decode(C.byref(desc), C.byref(w), fake[0], None, 1, 2, 103, fake[1],
                               fake[2], 64, C.byref(sel), None, fake[3], ws, 1024,
                               None) == dv.DV_ERR_WORKSPACE
    assert lib.dv_layer_decode(C.byref(desc), C.byref(w), fake[0], None, 1, 2, 103, fake[1],
                               fake[2], 64, C.byref(sel), None, fake[3], C.c_void_p(0x200010),
                               1 << 30, None) == dv.DV_ERR_WORKSPACE
    # predictor / blocks
    assert lib.dv_predict_topk(C.byref(desc), C.byref(w), fake[0], 1, 0, 5, C.byref(sel), None,
                               None, ws, 1 << 30, None) == dv.DV_ERR_INVALID_ARG
    assert lib.dv_sparse_attn(C.byref(desc), C.byref(w), fake[0], 1, fake[1], fake[2], 0, fake[3],
                              fake[4], 3, fake[5], ws, 1 << 30, None) == dv.DV_ERR_INVALID_ARG
    assert lib.dv_sparse_mlp(C.byref(desc), C.byref(w), fake[0], 1, fake[1], fake[2], 5, fake[0],
                             ws, 1 << 30, None) == dv.DV_ERR_INVALID_ARG
    assert lib.dv_hbm_copy(fake[0], fake[1], 17, None) == dv.DV_ERR_INVALID_ARG
    unsupported = dv.make_desc(256, 8, 24, 1024, 32, dv.DV_F32, 65)
    assert lib.dv_layer_decode(C.byref(unsupported), C.byref(w), fake[0], None, 1, 2, 103, fake[1],
                               fake[2], 64, C.byref(sel), None, fake[3], ws, 1 << 30,
                               None) == dv.DV_ERR_UNSUPPORTED


def test_row_kernel_variant_switch(dv):
    """Host-only: the variant switch accepts 0 and 1 and refuses the rest."""
    with pytest.raises(dv.DvError) as e:
        dv.dv_set_row_kernel(2)
    assert e.value.status == dv.DV_ERR_INVALID_ARG
    dv.dv_set_row_kernel(1)
    dv.dv_set_row_kernel(0)
