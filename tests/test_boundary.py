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
    assert d == 64 * 32 * (16384 // 2048) * 130 * 4  # [B, Hq, splits of 2048 keys, Dv + 2] fp32
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
    assert dec(D=192, Dv=192) == fa.SDPA_ERR_UNSUPPORTED  # value dim 128 only
    assert dec(Hq=34, Hkv=2) == fa.SDPA_ERR_UNSUPPORTED  # group of 17: more than one 16-row tile
    assert dec(dt=fa.SDPA_E4M3) == fa.SDPA_ERR_UNSUPPORTED
    assert dec(max_kv=0) == fa.SDPA_ERR_INVALID


def test_new_entry_points_are_declared(lib):
    names = set(fa.declared_functions())
    assert {"sdpa_fwd_varlen", "sdpa_fwd_varlen_fp8", "sdpa_fwd_varlen_workspace_size", "sdpa_fwd_int8",
            "sdpa_fwd_int8_workspace_size", "sdpa_fwd_host", "sdpa_fwd_host_workspace_size",
            "sdpa_decode_paged", "sdpa_decode_noalloc"} <= names


def test_new_workspace_sizes(lib):
    # packed sequences: the int32 tile prefix [B + 1], rounded up to 16 bytes
    assert fa.sdpa_fwd_varlen_workspace_size(1) == 16
    assert fa.sdpa_fwd_varlen_workspace_size(16) == 80
    assert fa.sdpa_fwd_varlen_workspace_size(0) == 0
    # int8 codes: 16-bit copies of Q and K (and V when int8); no device here, so no split part
    q, kv = 2 * 4096 * 32 * 128 * 2, 2 * 4096 * 8 * 128 * 2
    assert fa.sdpa_fwd_int8_workspace_size(2, 32, 8, 4096, 4096, 128, False, True) == q + kv
    assert fa.sdpa_fwd_int8_workspace_size(2, 32, 8, 4096, 4096, 128, True, True) == q + 2 * kv
    # host-buffer call: device copies of Q, K, V, O and LSE
    lse = 2 * 32 * 4096 * 4
    assert fa.sdpa_fwd_host_workspace_size(2, 32, 8, 4096, 4096, 128, 128, True) == q + 2 * kv + q + lse


def test_varlen_int8_and_host_validation_codes(lib):
    f, sz = ctypes.c_float, ctypes.c_size_t

    def varlen(**over):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cq=FAKE, ck=FAKE, B=2, Hq=4, Hkv=2, tq=100, tk=100,
                 maxq=60, D=128, Dv=128, strides=None, scale=f(0.1), causal=1, ws=FAKE, wsb=sz(1 << 10),
                 dt=fa.SDPA_BF16, odt=fa.SDPA_BF16, stream=None)
        a.update(over)
        return lib.sdpa_fwd_varlen(*a.values())

    assert varlen(B=0) == fa.SDPA_ERR_INVALID
    assert varlen(tk=0) == fa.SDPA_ERR_INVALID
    assert varlen(maxq=101) == fa.SDPA_ERR_INVALID     # longer than all the packed rows
    assert varlen(cq=None) == fa.SDPA_ERR_INVALID
    assert varlen(ck=ctypes.c_void_p(0x10002)) == fa.SDPA_ERR_INVALID  # offsets must be 4-byte aligned
    assert varlen(ws=None) == fa.SDPA_ERR_INVALID
    assert varlen(wsb=sz(8)) == fa.SDPA_ERR_INVALID      # below the tile prefix size
    assert varlen(dt=fa.SDPA_E4M3) == fa.SDPA_ERR_UNSUPPORTED
    assert varlen(D=96, Dv=96) == fa.SDPA_ERR_UNSUPPORTED

    def int8(**over):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, Sq=64, Sk=64, D=128, strides=None,
                 qs=FAKE, ks=FAKE, vs=None, scale=f(0.1), causal=1, ws=FAKE, wsb=sz(1 << 24),
                 vdt=fa.SDPA_F16, odt=fa.SDPA_F16, stream=None)
        a.update(over)
        return lib.sdpa_fwd_int8(*a.values())

    assert int8(qs=None) == fa.SDPA_ERR_INVALID
    assert int8(vs=FAKE) == fa.SDPA_ERR_INVALID           # 16-bit V takes no channel scales
    assert int8(vdt=fa.SDPA_I8) == fa.SDPA_ERR_INVALID    # int8 V needs them
    assert int8(vdt=fa.SDPA_BF16) == fa.SDPA_ERR_UNSUPPORTED  # V values in another type than O
    assert int8(odt=fa.SDPA_E4M3, vdt=fa.SDPA_E4M3) == fa.SDPA_ERR_UNSUPPORTED
    assert int8(D=192) == fa.SDPA_ERR_UNSUPPORTED         # head dims 64 and 128 only
    assert int8(wsb=sz(16)) == fa.SDPA_ERR_INVALID        # below the 16-bit copies
    assert int8(ks=ctypes.c_void_p(0x10002)) == fa.SDPA_ERR_INVALID

    def host(**over):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, Sq=64, Sk=64, D=128, Dv=128,
                 scale=f(0.1), causal=1, ws=FAKE, wsb=sz(1 << 24), dt=fa.SDPA_BF16, odt=fa.SDPA_BF16, stream=None)
        a.update(over)
        return lib.sdpa_fwd_host(*a.values())

    assert host(q=None) == fa.SDPA_ERR_INVALID
    assert host(Hkv=3) == fa.SDPA_ERR_INVALID
    assert host(wsb=sz(1024)) == fa.SDPA_ERR_INVALID
    assert host(odt=fa.SDPA_F16) == fa.SDPA_ERR_UNSUPPORTED
    assert host(dt=fa.SDPA_E4M3, odt=fa.SDPA_E4M3) == fa.SDPA_ERR_UNSUPPORTED
    assert host(D=96, Dv=96) == fa.SDPA_ERR_UNSUPPORTED
