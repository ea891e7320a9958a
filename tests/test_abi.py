"""The C-ABI library loads, exports every entry point include/moe_decode.h
declares, and rejects bad arguments on the host before any launch. No
compute call runs here (this suite also runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_decode.h")


@pytest.fixture(scope="module")
def api():
    from moe_decode_gb300 import build
    build.build()
    from moe_decode_gb300 import api as a
    return a


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("moe_route", "moe_ffn", "moe_decode_layer", "moe_workspace_bytes", "moe_read_status",
              "moe_status_str", "moe_workspace_init"):
        assert f in names


def test_library_exports_every_declared_symbol(api):
    lib = ctypes.CDLL(api.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_bytes_and_shape_checks(api):
    ling = api.make_shape(2560, 512, 8, 768, 768, 0)
    n1 = api.workspace_bytes(ling, 1)
    n2 = api.workspace_bytes(ling, 2)
    n16 = api.workspace_bytes(ling, 16)
    assert 0 < n2 < n16
    assert n16 >= 1024 + 16 * 512 * 4 + 16 * 768 * 2 + 16 * 8 * 768 * 2
    # one token: room for the split-K layer's partial outputs (MOE_MAX_GRID x H fp32)
    # and for the tagged activations (32-bit words, shared expert + k routed pairs)
    assert n1 >= 1024 + 512 * 8 + 256 * 2560 * 4 + (768 + 8 * 768) * 4
    mx1 = api.workspace_bytes(api.make_shape(2560, 512, 8, 768, 768, 1), 1)
    assert 0 < mx1 < n1  # MXFP4 one-token layers keep grid barrier 2: no tagged words
    assert api.workspace_bytes(ling, 0) == 0
    assert api.workspace_bytes(ling, 17) == 0
    for bad in (api.make_shape(2500, 512, 8, 768, 768),   # H not a multiple of 256
                api.make_shape(2560, 512, 17, 768, 768),  # k > 16
                api.make_shape(2560, 4, 8, 768, 768),     # k > E
                api.make_shape(2560, 2048, 8, 768, 768),  # E > 1024
                api.make_shape(2560, 512, 8, 700, 768),   # I % 64
                api.make_shape(2560, 512, 8, 768, 768, 3),  # no such format
                api.make_shape(2560, 512, 8, 704, 768, 2),  # FP8 needs I % 128
                api.make_shape(2816, 512, 8, 768, 768, 2),  # FP8 needs H % 512
                api.make_shape(256, 16, 2, 64, 64, 1)):   # MXFP4 needs H % 512
        assert api.workspace_bytes(bad, 1) == 0


def test_host_side_errors_before_launch(api):
    lib = api.lib
    s = api.make_shape(256, 16, 2, 64, 64, 0)
    P = ctypes.c_void_p
    fake = P(4096)
    assert lib.moe_route(fake, 0, fake, ctypes.byref(s), fake, fake, fake, 1 << 20, None) == api.EM
    assert lib.moe_route(None, 1, fake, ctypes.byref(s), fake, fake, fake, 1 << 20, None) == api.EINVAL
    assert lib.moe_route(P(4097), 1, fake, ctypes.byref(s), fake, fake, fake, 1 << 20, None) == api.EALIGN
    w = api._Weights(4096, 4096, 4096, None, None, None, 4096, 4096, 4096)
    assert lib.moe_decode_layer(fake, 1, fake, ctypes.byref(w), ctypes.byref(s), None, None, fake, fake,
                                1 << 20, 1 << 20, None) == api.EINVAL          # unknown flag
    w_missing = api._Weights(4096, None, 4096, None, None, None, 4096, 4096, 4096)
    assert lib.moe_ffn(fake, 1, fake, fake, ctypes.byref(w_missing), ctypes.byref(s), fake, fake, 1 << 20,
                       None) == api.EINVAL
    assert lib.moe_mxfp4_dequant(fake, fake, 4, 48, fake, None) == api.ESHAPE
    assert lib.moe_set_option(99, 1) == api.EINVAL
    assert lib.moe_set_option(api.OPT_WAIT_TIMEOUT_NS, 0) == api.EINVAL
    # output layer: format, shape and workspace checks before any launch
    assert lib.moe_lm_head(fake, 1, fake, None, 10, 256, 1, fake, fake, 1024, 0, None) == api.ESHAPE
    assert lib.moe_lm_head(fake, 1, fake, None, 10, 264, 2, fake, fake, 1024, 0, None) == api.ESHAPE
    assert lib.moe_lm_head(fake, 1, fake, None, 10, 256, 2, fake, fake, 1024, 0, None) == api.EINVAL
    assert lib.moe_lm_head(fake, 17, fake, None, 10, 256, 0, fake, fake, 1024, 0, None) == api.EM
    assert lib.moe_lm_head(fake, 1, fake, None, 10, 256, 0, fake, fake, 512, 0, None) == api.EWORKSPACE
    assert lib.moe_fp8_quantize(fake, 4, 100, 32, fake, fake, None) == api.ESHAPE
    assert api.status_str(api.ETIMEOUT).startswith("device")
    assert api.last_launch_count() == 0
