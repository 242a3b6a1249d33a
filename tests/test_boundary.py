"""CPU-side checks of the C ABI: the library loads, exports every declared symbol, and rejects
bad arguments with status codes before making any CUDA call."""
import ctypes

import pytest

import flash_attention_forward_gb300 as fa
from flash_attention_forward_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return fa.library()


def test_every_declared_function_is_exported(lib):
    names = fa.declared_functions()
    assert {"sdpa_fwd", "sdpa_fwd_fp8", "sdpa_decode", "sdpa_decode_workspace_size", "sdpa_fwd_workspace_size",
            "sdpa_check_device_status", "sdpa_status_string", "sdpa_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert fa.sdpa_status_string(fa.SDPA_OK) == "SDPA_OK"
    assert fa.sdpa_status_string(fa.SDPA_ERR_TIMEOUT) == "SDPA_ERR_TIMEOUT"
    assert fa.sdpa_status_string(99) == "SDPA_ERR_UNKNOWN"
    assert fa.sdpa_version() >= 100


def test_workspace_sizes(lib):
    # no GPU here: the device-dependent split part is zero, only the condensed mask remains
    assert fa.sdpa_fwd_workspace_size(3, 28, 1000, 3001, 128, False, False) == 0
    n = fa.sdpa_fwd_workspace_size(3, 28, 1000, 3001, 128, False, True)
    rows, nkb = 3 * 1000, (3001 + 127) // 128
    assert n >= rows * nkb * 17 and n % 16 == 0
    assert fa.sdpa_fwd_workspace_size(0, 28, 1000, 3001, 128, False, True) == 0
    d = fa.sdpa_decode_workspace_size(64, 32, 16384, 128)
    assert d == 64 * 32 * 16 * 130 * 4
    assert fa.sdpa_decode_workspace_size(0, 32, 16384, 128) == 0


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation first


def _fwd(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, Sq=16, Sk=16, D=128, Dv=128,
             strides=None, scale=0.1, causal=0, mask=None, mstr=None, ws=None, wsb=0, dt=fa.SDPA_BF16,
             odt=fa.SDPA_BF16, stream=None)
    a.update(over)
    return lib.sdpa_fwd(*a.values())


def test_fwd_validation_codes(lib):
    assert _fwd(lib, q=None) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, o=None) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, Hkv=3) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, Sq=0) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, Sk=-1) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, scale=0.0) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, scale=float("nan")) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, scale=float("inf")) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, D=96, Dv=96) == fa.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, D=128, Dv=64) == fa.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, dt=fa.SDPA_E4M3) == fa.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, odt=fa.SDPA_F16) == fa.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, q=ctypes.c_void_p(0x10008)) == fa.SDPA_ERR_UNSUPPORTED  # not 16-byte aligned
    bad = (ctypes.c_int64 * 12)(16 * 4 * 128, 4 * 128 + 4, 128, 0, 0, 0, 0, 0, 0, 0, 0, 0)
    assert _fwd(lib, strides=bad) == fa.SDPA_ERR_UNSUPPORTED
    # a mask needs a large enough, aligned workspace
    assert _fwd(lib, mask=FAKE) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, mask=FAKE, ws=FAKE, wsb=15) == fa.SDPA_ERR_INVALID
    assert _fwd(lib, mask=ctypes.c_void_p(0x10001), ws=FAKE, wsb=1 << 20) == fa.SDPA_ERR_INVALID


def test_fp8_and_decode_validation_codes(lib):
    f = ctypes.c_float
    # e4m3: bad descale, unsupported head dims, unsupported output dtype
    args = [FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 16, 16, 192, 128, None, f(0.1), 1, None, None, None, 0]
    assert lib.sdpa_fwd_fp8(*args, f(0.0), f(1.0), f(1.0), fa.SDPA_BF16, None) == fa.SDPA_ERR_INVALID
    assert lib.sdpa_fwd_fp8(*args, f(1.0), f(1.0), f(1.0), fa.SDPA_F16, None) == fa.SDPA_ERR_UNSUPPORTED
    args[10] = 64
    assert lib.sdpa_fwd_fp8(*args, f(1.0), f(1.0), f(1.0), fa.SDPA_BF16, None) == fa.SDPA_ERR_UNSUPPORTED

    def dec(**over):
        a = dict(q=FAKE, k=FAKE, v=FAKE, kv=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, max_kv=100, D=128, Dv=128,
                 strides=None, scale=0.1, ws=FAKE, wsb=1 << 20, dt=fa.SDPA_BF16, stream=None)
        a.update(over)
        return lib.sdpa_decode(*a.values())

    assert dec(kv=None) == fa.SDPA_ERR_INVALID
    assert dec(ws=None) == fa.SDPA_ERR_INVALID
    assert dec(wsb=100) == fa.SDPA_ERR_INVALID
    assert dec(Hkv=3) == fa.SDPA_ERR_INVALID
    assert dec(D=64, Dv=64) == fa.SDPA_ERR_UNSUPPORTED
    assert dec(Hq=32, Hkv=2) == fa.SDPA_ERR_UNSUPPORTED  # group of 16
    assert dec(dt=fa.SDPA_E4M3) == fa.SDPA_ERR_UNSUPPORTED
    assert dec(max_kv=0) == fa.SDPA_ERR_INVALID
