"""The C ABI without a GPU: the library builds and loads, exports every entry
point ``include/moe_w4a16.h`` declares, and rejects bad arguments on the host
before anything is launched."""
import ctypes
import os
import re

import pytest

import quantized_moe_expert_align_gb300 as moe
from quantized_moe_expert_align_gb300 import build

HEADER = os.path.join(build.INCLUDE, "moe_w4a16.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)) - {"moe_stream_t"})


def test_header_declares_the_entry_points():
    names = declared_functions()
    for need in ["moe_w4a16_prepack", "moe_align", "moe_w4a16_forward",
                 "moe_w4a16_workspace_size", "moe_status_string"]:
        assert need in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported by {moe.LIB_PATH}"


def test_status_strings(lib):
    for code in range(11):
        s = moe.moe_status_string(code)
        assert s.startswith("MOE_")
    assert moe.moe_status_string(0) == "MOE_OK"
    assert "UNKNOWN" in moe.moe_status_string(99)


def test_prepack_size(lib):
    st, b = moe.moe_w4a16_prepack_size(moe.MOE_PACK_W13, 384, 4096, 7168, 32)
    assert st == moe.MOE_OK
    # header + int4 codes + one fp16 scale per 32 weights
    assert b == 256 + 384 * 4096 * 7168 // 2 + 384 * 4096 * (7168 // 32) * 2
    # wider scale groups are stored in the same layout: same size
    for g in (64, 128):
        st, b2 = moe.moe_w4a16_prepack_size(moe.MOE_PACK_W13, 384, 4096, 7168, g)
        assert st == moe.MOE_OK and b2 == b
    for bad in [(3, 8, 256, 256, 32), (1, 8, 256, 256, 16), (1, 8, 256, 256, 96),
                (1, 8, 256, 256, 256), (1, 0, 256, 256, 32),
                (1, 8, 200, 256, 32), (1, 8, 256, 96, 32)]:
        st, b = moe.moe_w4a16_prepack_size(*bad)
        assert st == moe.MOE_ERR_INVALID_ARG and b == 0


def test_workspace_sizes(lib):
    assert moe.moe_w4a16_workspace_size(4, 2, 8, 256, 128) > 0
    small = moe.moe_w4a16_workspace_size(1, 8, 384, 7168, 2048)
    big = moe.moe_w4a16_workspace_size(90, 8, 384, 7168, 2048)
    assert 0 < small < big
    assert moe.moe_w4a16_workspace_size(0, 8, 384, 7168, 2048) > 0
    for bad in [(-1, 8, 384, 7168, 2048), (1, 0, 384, 7168, 2048), (1, 65, 384, 7168, 2048),
                (1, 8, 0, 7168, 2048), (1, 8, 2000, 7168, 2048), (1, 8, 384, 7000, 2048),
                (1, 8, 384, 7168, 2000)]:
        assert moe.moe_w4a16_workspace_size(*bad) == 0
    assert moe.moe_align_workspace_size(1, 8, 384) >= 256
    assert moe.moe_align_workspace_size(1, 8, 1025) == 0


def _fwd(lib, **kw):
    args = dict(hidden=4096, ids=4096, w=4096, w13=4096, w2=4096, out=4096,
                M=4, k=2, E=8, H=256, I=128, ws=4096, ws_bytes=1 << 30)
    args.update(kw)
    return lib.moe_w4a16_forward(args["hidden"], args["ids"], args["w"], args["w13"], args["w2"],
                                 args["out"], args["M"], args["k"], args["E"], args["H"],
                                 args["I"], args["ws"], args["ws_bytes"], None)


def test_forward_host_validation(lib):
    assert _fwd(lib, w13=None) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, hidden=None) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, H=250) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, I=96) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, k=0) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, E=0) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, M=-1) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(lib, hidden=4104) == moe.MOE_ERR_MISALIGNED
    assert _fwd(lib, out=4100) == moe.MOE_ERR_MISALIGNED
    assert _fwd(lib, w2=4112) == moe.MOE_ERR_MISALIGNED
    assert _fwd(lib, ws=4160) == moe.MOE_ERR_MISALIGNED
    assert _fwd(lib, ws_bytes=1024) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    # M == 0 may pass null token pointers; it still needs a device to say OK
    st = _fwd(lib, M=0, hidden=None, ids=None, w=None, out=None)
    assert st in (moe.MOE_OK, moe.MOE_ERR_UNSUPPORTED_DEVICE)


def test_align_and_prepack_host_validation(lib):
    p = 4096
    assert lib.moe_align(p, 4, 2, 0, p, p, p, p, p, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_align(None, 4, 2, 8, p, p, p, p, p, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_align(p, 4, 2, 8, p, p, p, p, p + 8, 1 << 20, None) == moe.MOE_ERR_MISALIGNED
    assert lib.moe_align(p, 4, 2, 8, p, p, p, p, p, 16, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_w4a16_prepack(1, p, p, 8, 256, 256, 32, p, 16, None) == \
        moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_w4a16_prepack(1, p + 4, p, 8, 256, 256, 32, p, 1 << 30, None) == \
        moe.MOE_ERR_MISALIGNED
    assert lib.moe_w4a16_prepack(1, p, p, 8, 256, 256, 32, p + 16, 1 << 30, None) == \
        moe.MOE_ERR_MISALIGNED
    assert lib.moe_w4a16_prepack(1, None, p, 8, 256, 256, 32, p, 1 << 30, None) == \
        moe.MOE_ERR_INVALID_ARG


def test_router_host_validation(lib):
    p = 4096
    ra = lib.moe_route_align
    args = [p, 4, 2, 8, p, p, p, p, p, p, p, 1 << 20, None]

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return ra(*a)
    assert call(a3=1) == moe.MOE_ERR_INVALID_ARG           # k > E
    assert call(a2=0) == moe.MOE_ERR_INVALID_ARG           # k = 0
    assert call(a0=None) == moe.MOE_ERR_INVALID_ARG        # logits
    assert call(a5=None) == moe.MOE_ERR_INVALID_ARG        # topk_w
    assert call(a0=p + 2) == moe.MOE_ERR_MISALIGNED
    assert call(a10=p + 64) == moe.MOE_ERR_MISALIGNED      # workspace
    assert call(a11=16) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    fr = lib.moe_w4a16_forward_routed
    good = [p, p, p, p, p, p, p, 4, 2, 8, 256, 128, p, 1 << 30, None]
    bad = list(good)
    bad[1] = None
    assert fr(*bad) == moe.MOE_ERR_INVALID_ARG             # logits
    bad = list(good)
    bad[8], bad[9] = 9, 8
    assert fr(*bad) == moe.MOE_ERR_INVALID_ARG             # k > E
    bad = list(good)
    bad[1] = p + 1
    assert fr(*bad) == moe.MOE_ERR_MISALIGNED


def test_no_gpu_reports_unsupported_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib) == moe.MOE_ERR_UNSUPPORTED_DEVICE


def test_diag_starts_at_version_2(lib):
    d = moe.moe_w4a16_get_diag()
    assert d["version"] == 2 and d["reserved"] == 0
