"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host with the documented
status codes (no CUDA call is reached by any of these)."""
import ctypes
import os
import re

import pytest

import paged_fp8_kv_03_gb300 as pkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedfp8.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def _status_codes():
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"(PKV_ERR_[A-Z]+|PKV_OK)\s*=\s*(\d+)", text)}


@pytest.fixture(scope="module")
def lib():
    return pkv.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"pkv_kv_append_fp8", "pkv_paged_gqa_decode", "pkv_decode_workspace_size",
            "pkv_status_string", "pkv_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    codes = _status_codes()
    assert codes["PKV_OK"] == 0 and len(codes) == 8
    for name, c in codes.items():
        s = pkv.pkv_status_string(c)
        assert s and s != "unknown status", name
    assert pkv.pkv_status_string(12345) == "unknown status"
    assert pkv.pkv_version() >> 16 == 1


A16 = ctypes.c_void_p(0x10000)      # fake, 16-byte-aligned addresses: never dereferenced on these paths
A16b = ctypes.c_void_p(0x20000)


def _append(lib, **kw):
    args = dict(k=A16, v=A16, dtype=0, T=4, H=8, D=128, slots=A16, ks=A16, vs=A16, kc=A16, vc=A16b,
                np_=10, P=16, err=None)
    args.update(kw)
    return lib.pkv_kv_append_fp8(args["k"], args["v"], args["dtype"], args["T"], args["H"], args["D"],
                                 args["slots"], args["ks"], args["vs"], args["kc"], args["vc"], args["np_"],
                                 args["P"], args["err"], None)


def test_append_argument_errors(lib):
    c = _status_codes()
    assert _append(lib, T=-1) == c["PKV_ERR_SHAPE"]
    assert _append(lib, H=0) == c["PKV_ERR_SHAPE"]
    assert _append(lib, np_=0) == c["PKV_ERR_SHAPE"]
    assert _append(lib, dtype=7) == c["PKV_ERR_DTYPE"]
    assert _append(lib, D=64) == c["PKV_ERR_UNSUPPORTED"]
    assert _append(lib, P=8) == c["PKV_ERR_UNSUPPORTED"]
    assert _append(lib, P=48) == c["PKV_ERR_UNSUPPORTED"]
    assert _append(lib, P=512) == c["PKV_ERR_UNSUPPORTED"]
    assert _append(lib, k=None) == c["PKV_ERR_NULL"]
    assert _append(lib, slots=None) == c["PKV_ERR_NULL"]
    assert _append(lib, kc=ctypes.c_void_p(0x10008)) == c["PKV_ERR_ALIGN"]
    assert _append(lib, k=ctypes.c_void_p(0x10004)) == c["PKV_ERR_ALIGN"]
    assert _append(lib, err=ctypes.c_void_p(0x10002)) == c["PKV_ERR_ALIGN"]
    assert _append(lib, T=0, k=None, v=None, slots=None) == c["PKV_OK"]     # empty append is a no-op


def _decode(lib, **kw):
    a = dict(q=A16, kc=A16, vc=A16b, ks=A16, vs=A16, bt=A16, maxp=4, lens=A16, maxl=0, psz=None, B=2, Hq=16,
             Hkv=2, D=128, P=16, np_=8, sm=0.088, out=A16, odt=1, ws=A16, wsb=1 << 20, err=None, ctas=0)
    a.update(kw)
    return lib.pkv_paged_gqa_decode(a["q"], a["kc"], a["vc"], a["ks"], a["vs"], a["bt"], a["maxp"], a["lens"],
                                    a["maxl"], a["psz"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"], a["np_"],
                                    a["sm"], a["out"], a["odt"], a["ws"], a["wsb"], a["err"], a["ctas"], None)


def test_decode_argument_errors(lib):
    c = _status_codes()
    assert _decode(lib, Hq=12, Hkv=8) == c["PKV_ERR_SHAPE"]          # Hq % Hkv
    assert _decode(lib, B=-1) == c["PKV_ERR_SHAPE"]
    assert _decode(lib, maxp=0) == c["PKV_ERR_SHAPE"]
    assert _decode(lib, np_=0) == c["PKV_ERR_SHAPE"]
    assert _decode(lib, Hq=32, Hkv=2) == c["PKV_ERR_UNSUPPORTED"]    # G = 16
    assert _decode(lib, D=64) == c["PKV_ERR_UNSUPPORTED"]
    assert _decode(lib, P=48) == c["PKV_ERR_UNSUPPORTED"]
    assert _decode(lib, P=512) == c["PKV_ERR_UNSUPPORTED"]
    assert _decode(lib, B=pkv.MAX_BATCH + 1) == c["PKV_ERR_UNSUPPORTED"]
    assert _decode(lib, np_=1 << 30, Hkv=2) == c["PKV_ERR_UNSUPPORTED"]   # tile index would overflow int32
    assert _decode(lib, odt=5) == c["PKV_ERR_DTYPE"]
    assert _decode(lib, sm=float("nan")) == c["PKV_ERR_SHAPE"]
    assert _decode(lib, sm=float("inf")) == c["PKV_ERR_SHAPE"]
    assert _decode(lib, q=None) == c["PKV_ERR_NULL"]
    assert _decode(lib, bt=None) == c["PKV_ERR_NULL"]
    assert _decode(lib, out=None) == c["PKV_ERR_NULL"]
    assert _decode(lib, kc=ctypes.c_void_p(0x10001)) == c["PKV_ERR_ALIGN"]
    assert _decode(lib, out=ctypes.c_void_p(0x10008)) == c["PKV_ERR_ALIGN"]
    assert _decode(lib, ws=None) == c["PKV_ERR_WORKSPACE"]
    assert _decode(lib, ws=ctypes.c_void_p(0x10010)) == c["PKV_ERR_WORKSPACE"]
    assert _decode(lib, B=0, q=None, bt=None, lens=None, out=None) == c["PKV_OK"]
    assert _decode(lib, maxl=-1) == c["PKV_ERR_SHAPE"]
    assert _decode(lib, psz=ctypes.c_void_p(0x10002)) == c["PKV_ERR_ALIGN"]
    assert _decode(lib, psz=A16, maxp=1 << 24) == c["PKV_ERR_UNSUPPORTED"]   # max_pages * 256 overflows int32


def test_workspace_size_rejects_unsupported(lib):
    assert pkv.pkv_decode_workspace_size(2, 12, 8) == 0
    assert pkv.pkv_decode_workspace_size(2, 16, 8, head_dim=64) == 0
    assert pkv.pkv_decode_workspace_size(2, 16, 8, page_size=8) == 0
    assert pkv.pkv_decode_workspace_size(2, 16, 8, max_seq_len=-1) == 0


def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 128)
    with pytest.raises(ValueError):
        pkv.pkv_kv_append_fp8(x, x, torch.zeros(1, dtype=torch.int64), torch.ones(1), torch.ones(1),
                              torch.zeros(1, 1, 16, 128, dtype=torch.uint8),
                              torch.zeros(1, 1, 16, 128, dtype=torch.uint8))


def _fused(lib, **kw):
    a = dict(kn=A16, vn=A16, dt=0, n=1, q=A16, kc=A16, vc=A16b, ks=A16, vs=A16, bt=A16, maxp=4, lens=A16, maxl=0,
             psz=None, B=2, Hq=16, Hkv=2, D=128, P=16, np_=8, sm=0.088, out=A16, odt=1, ws=A16, wsb=1 << 20,
             err=None, ctas=0)
    a.update(kw)
    return lib.pkv_append_decode_fp8(a["kn"], a["vn"], a["dt"], a["n"], a["q"], a["kc"], a["vc"], a["ks"], a["vs"],
                                     a["bt"], a["maxp"], a["lens"], a["maxl"], a["psz"], a["B"], a["Hq"], a["Hkv"],
                                     a["D"], a["P"], a["np_"], a["sm"], a["out"], a["odt"], a["ws"], a["wsb"],
                                     a["err"], a["ctas"], None)


def test_fused_argument_errors(lib):
    c = _status_codes()
    assert _fused(lib, n=-1) == c["PKV_ERR_SHAPE"]
    assert _fused(lib, dt=9) == c["PKV_ERR_DTYPE"]
    assert _fused(lib, kn=None) == c["PKV_ERR_NULL"]
    assert _fused(lib, vn=ctypes.c_void_p(0x10004)) == c["PKV_ERR_ALIGN"]
    assert _fused(lib, Hq=12, Hkv=8) == c["PKV_ERR_SHAPE"]
    assert _fused(lib, P=24) == c["PKV_ERR_UNSUPPORTED"]
    assert _fused(lib, B=0, kn=None, vn=None, q=None, bt=None, lens=None, out=None) == c["PKV_OK"]


def test_calibrate_argument_errors(lib):
    c = _status_codes()

    def cal(**kw):
        a = dict(k=A16, v=A16, dt=0, T=4, H=8, D=128, rk=A16, rv=A16b, ks=A16, vs=A16b)
        a.update(kw)
        return lib.pkv_kv_calibrate(a["k"], a["v"], a["dt"], a["T"], a["H"], a["D"], a["rk"], a["rv"], a["ks"],
                                    a["vs"], None)
    assert cal(T=-1) == c["PKV_ERR_SHAPE"]
    assert cal(H=0) == c["PKV_ERR_SHAPE"]
    assert cal(dt=4) == c["PKV_ERR_DTYPE"]
    assert cal(D=96) == c["PKV_ERR_UNSUPPORTED"]
    assert cal(rk=None) == c["PKV_ERR_NULL"]
    assert cal(ks=None) == c["PKV_ERR_NULL"]          # both scales or neither
    assert cal(k=None) == c["PKV_ERR_NULL"]
    assert cal(k=ctypes.c_void_p(0x10008)) == c["PKV_ERR_ALIGN"]


def test_prefill_argument_errors(lib):
    c = _status_codes()

    def pre(**kw):
        a = dict(q=A16, cu=A16, T=64, mq=32, kc=A16, vc=A16b, ks=A16, vs=A16, bt=A16, maxp=4, lens=A16, psz=None,
                 B=2, mkv=64, mtot=0, Hq=16, Hkv=2, D=128, P=16, np_=8, sm=0.088, out=A16, odt=1, ws=A16,
                 wsb=1 << 24, err=None)
        a.update(kw)
        return lib.pkv_paged_prefill(a["q"], a["cu"], a["T"], a["mq"], a["kc"], a["vc"], a["ks"], a["vs"],
                                     a["bt"], a["maxp"], a["lens"], a["psz"], a["B"], a["mkv"], a["mtot"], a["Hq"],
                                     a["Hkv"], a["D"], a["P"], a["np_"], a["sm"], a["out"], a["odt"], a["ws"],
                                     a["wsb"], a["err"], None)
    assert pre(T=-1) == c["PKV_ERR_SHAPE"]
    assert pre(mq=-1) == c["PKV_ERR_SHAPE"]
    assert pre(mkv=-1) == c["PKV_ERR_SHAPE"]
    assert pre(Hq=12, Hkv=8) == c["PKV_ERR_SHAPE"]
    assert pre(maxp=0) == c["PKV_ERR_SHAPE"]
    assert pre(sm=float("nan")) == c["PKV_ERR_SHAPE"]
    assert pre(sm=0.0) == c["PKV_ERR_SHAPE"]
    assert pre(sm=-0.088) == c["PKV_ERR_SHAPE"]
    assert pre(odt=3) == c["PKV_ERR_DTYPE"]
    assert pre(D=64) == c["PKV_ERR_UNSUPPORTED"]
    assert pre(P=48) == c["PKV_ERR_UNSUPPORTED"]
    assert pre(Hq=32, Hkv=2) == c["PKV_ERR_UNSUPPORTED"]             # G = 16
    assert pre(B=8192, Hkv=2, Hq=16, mq=1 << 30) == c["PKV_ERR_UNSUPPORTED"]   # grid above 2^31
    assert pre(cu=None) == c["PKV_ERR_NULL"]
    assert pre(q=None) == c["PKV_ERR_NULL"]
    assert pre(q=ctypes.c_void_p(0x10008)) == c["PKV_ERR_ALIGN"]
    assert pre(cu=ctypes.c_void_p(0x10002)) == c["PKV_ERR_ALIGN"]
    assert pre(out=ctypes.c_void_p(0x10004)) == c["PKV_ERR_ALIGN"]
    assert pre(ws=None) == c["PKV_ERR_WORKSPACE"]
    assert pre(ws=ctypes.c_void_p(0x10010)) == c["PKV_ERR_WORKSPACE"]          # not 256-byte aligned
    need = pkv.pkv_prefill_workspace_size(2, 2, 64)
    assert need == 256 + 2 * 2 * 2 * 128 * 128 * 2                              # offsets, then K and V rows padded to 128
    assert pre(wsb=need - 1) == c["PKV_ERR_WORKSPACE"]
    # a bound on the lengths' sum shrinks the copies: 3 sequences of up to 128K, 130K tokens in all
    assert pkv.pkv_prefill_workspace_size(3, 8, 131072, 133120) == 256 + 2 * 8 * (1040 + 3) * 128 * 128 * 2
    assert pkv.pkv_prefill_workspace_size(3, 8, 131072) == 256 + 2 * 8 * 3 * 1024 * 128 * 128 * 2
    assert pre(mtot=-1) == c["PKV_ERR_SHAPE"]
    assert pre(psz=ctypes.c_void_p(0x10001)) == c["PKV_ERR_ALIGN"]
    assert pre(T=0, q=None, cu=None, out=None) == c["PKV_OK"]          # nothing to compute
    assert pre(mq=0, q=None, cu=None, out=None) == c["PKV_OK"]
    assert pkv.pkv_prefill_workspace_size(-1, 2, 64) == 0
    assert pkv.pkv_prefill_workspace_size(2, 2, 64, -5) == 0


def test_read_device_error_argument_errors(lib):
    c = _status_codes()
    code = ctypes.c_int32(0)
    assert lib.pkv_read_device_error(None, 0, ctypes.byref(code), None) == c["PKV_ERR_NULL"]
    assert lib.pkv_read_device_error(A16, 0, None, None) == c["PKV_ERR_NULL"]
    assert lib.pkv_read_device_error(ctypes.c_void_p(0x10002), 1, ctypes.byref(code), None) == c["PKV_ERR_ALIGN"]


def test_withhold_facility_is_off_at_load_and_settable(lib):
    lib.pkv_test_withhold_load(-5)          # any negative index turns it off
    lib.pkv_test_withhold_load(-1)


def test_split_weight_argument_errors(lib):
    """Weights outside [768, 1280], more than 1024 CTAs or a NULL array are
    rejected before any CUDA call; so are calibration requests with no
    rounds or no sequences."""
    c = _status_codes()
    ok = (ctypes.c_uint16 * 4)(768, 1024, 1100, 1280)
    low = (ctypes.c_uint16 * 4)(768, 767, 1024, 1024)
    high = (ctypes.c_uint16 * 4)(1024, 1281, 1024, 1024)
    assert lib.pkv_decode_set_split_weights(ctypes.addressof(low), 4) == c["PKV_ERR_SHAPE"]
    assert lib.pkv_decode_set_split_weights(ctypes.addressof(high), 4) == c["PKV_ERR_SHAPE"]
    assert lib.pkv_decode_set_split_weights(ctypes.addressof(ok), -1) == c["PKV_ERR_SHAPE"]
    assert lib.pkv_decode_set_split_weights(ctypes.addressof(ok), 1025) == c["PKV_ERR_SHAPE"]
    assert lib.pkv_decode_set_split_weights(None, 4) == c["PKV_ERR_NULL"]
    assert lib.pkv_decode_get_split_weights(ctypes.addressof(ok), 4, None) == c["PKV_ERR_NULL"]
    n = ctypes.c_int(0)
    assert lib.pkv_decode_get_split_weights(None, 4, ctypes.byref(n)) == c["PKV_ERR_NULL"]

    def cal(rounds=4, B=2):
        return lib.pkv_decode_calibrate_split(A16, A16, A16b, A16, A16, A16, 8, A16, 0, None, B, 16, 8, 128, 16, 100,
                                              0.088, A16, 0, A16, 1 << 20, 0, rounds, None, 0, None, None)
    assert cal(rounds=0) == c["PKV_ERR_SHAPE"]
    assert cal(rounds=65) == c["PKV_ERR_SHAPE"]
    assert cal(B=0) == c["PKV_ERR_SHAPE"]
