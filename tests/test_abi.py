"""The C-ABI library without a GPU: it builds, loads, exports every function
that include/moe.h declares, and rejects bad arguments on the host before
launching anything."""
import ctypes
import os
import re

import pytest

import aware_expert_routing_gb300 as moe
from aware_expert_routing_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(moe.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_no_cpu_fallback_when_library_missing(tmp_path):
    with pytest.raises(ImportError):
        moe.load(str(tmp_path / "libmissing.so"))


def P(**kw):
    base = dict(B=16, d=2048, N=128, k=8)
    base.update(kw)
    return moe.RouteParams(**base)


def test_slots_and_workspace(lib):
    assert moe.moe_num_slots(P()) == 8
    # router + routing (one cluster launch where the device allows it) + experts
    assert moe.moe_layer_launches(P(), 768) in (2, 3)
    assert moe.moe_layer_launches(P(B=0), 768) == 1            # the routing kernel only
    assert moe.moe_layer_launches(P(B=64), 768) == 3           # router, routing, experts
    assert moe.moe_layer_launches(P(dtype=moe.DTYPE_F32), 768) == 5   # router, routing, three fp32 expert kernels
    with pytest.raises(moe.MoeError):
        moe.moe_layer_launches(P(), 100)                       # d_ff not a multiple of 64
    assert moe.moe_num_slots(P(mode=moe.MODE_OEA, k0=3)) == 8
    assert moe.moe_num_slots(P(mode=moe.MODE_OEA, k0=3, kmax=11)) == 11
    a = moe.moe_workspace_bytes(P(), 768)
    b = moe.moe_workspace_bytes(P(), 0)
    assert a > b > 0 and a % 256 == 0
    # H (bf16, pairs x d_ff) and Y (fp32, pairs x d) dominate
    assert a >= 16 * 8 * 768 * 2 + 16 * 8 * 2048 * 4


@pytest.mark.parametrize("kw", [
    dict(B=257), dict(B=-1), dict(d=100), dict(d=32), dict(N=0), dict(N=1025), dict(k=0),
    dict(k=33, N=64), dict(k=9, N=8), dict(mode=2), dict(dtype=3),
    dict(mode=moe.MODE_OEA, k0=9), dict(mode=moe.MODE_OEA, k0=0, p=0.0),
    dict(mode=moe.MODE_OEA, k0=3, p=0.0), dict(mode=moe.MODE_OEA, k0=3, p=1.5),
    dict(mode=moe.MODE_OEA, k0=3, p=float("nan")),
    dict(mode=moe.MODE_OEA, k0=4, kmax=3), dict(mode=moe.MODE_OEA, k0=4, kmax=40),
    dict(B=4, B_valid=5),
])
def test_invalid_params_rejected_on_host(lib, kw):
    prm = P(**kw).c()
    assert lib.moe_num_slots(ctypes.byref(prm)) == -1
    assert lib.moe_workspace_bytes(ctypes.byref(prm), 768) == 0
    fake = ctypes.c_void_p(4096)
    r = moe._Routing(*([fake] * 7 + [None, None]))
    st = lib.moe_route(fake, fake, None, ctypes.byref(prm), ctypes.byref(r), fake, 1 << 30, None)
    assert st == moe.MOE_ERR_ARG


def test_bad_buffers_rejected_on_host(lib):
    prm = P().c()
    fake = ctypes.c_void_p(4096)
    r = moe._Routing(*([fake] * 7 + [None, None]))
    ws = moe.moe_workspace_bytes(P(), 768)
    # workspace too small, NULL, misaligned
    assert lib.moe_route(fake, fake, None, ctypes.byref(prm), ctypes.byref(r), fake, 16, None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_route(fake, fake, None, ctypes.byref(prm), ctypes.byref(r), None, ws, None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_route(fake, fake, None, ctypes.byref(prm), ctypes.byref(r), ctypes.c_void_p(4096 + 64), ws,
                         None) == moe.MOE_ERR_WORKSPACE
    # a NULL routing buffer, a misaligned hidden pointer
    r2 = moe._Routing(*([fake] * 6 + [None, None, None]))
    assert lib.moe_route(fake, fake, None, ctypes.byref(prm), ctypes.byref(r2), fake, ws, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(ctypes.c_void_p(4097), fake, None, ctypes.byref(prm), ctypes.byref(r), fake, ws,
                         None) == moe.MOE_ERR_ARG
    # d_ff not a multiple of 64
    assert lib.moe_expert_ffn(fake, fake, fake, fake, 100, ctypes.byref(prm), ctypes.byref(r), fake, fake, ws,
                              None) == moe.MOE_ERR_ARG
    assert b"d_ff" in lib.moe_last_error()
    assert lib.moe_status_string(moe.MOE_ERR_WORKSPACE) == b"MOE_ERR_WORKSPACE"


def test_batch_size_policy_is_accepted(lib):
    """k0 <= 0 in OEA mode chooses k0 from the batch instead of failing."""
    for B in (0, 1, 4, 16, 256):
        for k0 in (0, -3):
            assert moe.moe_num_slots(P(B=B, mode=moe.MODE_OEA, k0=k0, p=0.7)) == 8
    assert moe.moe_num_slots(P(mode=moe.MODE_OEA, k0=0, kmax=4)) == 4    # k0 = 3 at B = 16
    assert lib.moe_num_slots(ctypes.byref(P(B=4, mode=moe.MODE_OEA, k0=0, kmax=4).c())) == -1   # k0 = 5 > kmax


def test_int4_pack_checks_its_arguments(lib):
    fake = ctypes.c_void_p(4096)
    for rows, cols, rb, w, out in [(64, 100, 64, fake, fake), (64, 256, 48, fake, fake), (60, 256, 64, fake, fake),
                                   (64, 256, 64, None, fake), (64, 256, 64, fake, ctypes.c_void_p(4104))]:
        assert lib.moe_pack_int4(w, rows, cols, rb, out, None) == moe.MOE_ERR_ARG
    assert moe.int4_image_bytes(768, 2048) == 768 * 2048 // 2 + 768 * 16 * 2


def test_mixed_layer_checks_its_descriptor_before_launching(lib):
    """moe_decode_layer_mixed rejects a bad expert descriptor on the host,
    so not even the routing kernel is launched."""
    prm = P(mode=moe.MODE_OEA, k0=3).c()
    fake = ctypes.c_void_p(4096)
    r = moe._Routing(*([fake] * 7 + [None, None]))
    ws = moe.moe_workspace_bytes(P(mode=moe.MODE_OEA, k0=3), 768)
    bad = [moe._Mixed(None, fake, fake, fake, 32, 96),            # no slot table
           moe._Mixed(fake, ctypes.c_void_p(4100), fake, fake, 32, 96),   # misaligned image
           moe._Mixed(fake, fake, fake, fake, 0, 128),            # no bf16 expert
           moe._Mixed(fake, None, fake, fake, 32, 96)]            # missing image
    for m in bad:
        assert lib.moe_decode_layer_mixed(fake, fake, None, fake, fake, fake, ctypes.byref(m), 768,
                                          ctypes.byref(prm), ctypes.byref(r), fake, fake, ws, None) == moe.MOE_ERR_ARG
    assert lib.moe_decode_layer_mixed(fake, fake, None, fake, fake, fake, None, 768, ctypes.byref(prm),
                                      ctypes.byref(r), fake, fake, ws, None) == moe.MOE_ERR_ARG
    m = moe._Mixed(fake, fake, fake, fake, 32, 96)
    assert lib.moe_decode_layer_mixed(fake, fake, None, fake, fake, fake, ctypes.byref(m), 100,   # d_ff % 128
                                      ctypes.byref(prm), ctypes.byref(r), fake, fake, ws, None) == moe.MOE_ERR_ARG
