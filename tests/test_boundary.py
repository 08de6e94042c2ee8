"""The C-ABI boundary without a GPU: the library builds and loads, exports every
symbol include/kda.h declares, and rejects malformed arguments on the host with
the documented status codes.  Every call here carries at least one invalid
argument, so validation returns before anything touches a device (the fake
pointers are never dereferenced)."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_52_gb300 import build as kbuild
from gated_delta_rule_52_gb300 import kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    kbuild.build_library()
    return kda.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert set(declared_functions()) == set(kda.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert kda.lib().kda_version() >= 100
    for code in range(0, 11):
        s = kda.status_string(code)
        assert s.startswith("KDA_")
    assert "unknown" in kda.status_string(99)


# Fake, 16-byte aligned, never-dereferenced addresses.
P = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(12)]


def call(**over):
    a = dict(q=P[0], k=P[1], v=P[2], g=P[3], beta=P[4], scale=0.088, out=P[5], A_log=P[6],
             dt_bias=P[7], lb=-5.0, init=None, fin=None, sdt=0, cu=None, nseq=0,
             B=1, T=64, H=2, K=128, V=128, stream=None)
    a.update(over)
    return kda.raw_call(a["q"], a["k"], a["v"], a["g"], a["beta"], ctypes.c_float(a["scale"]),
                        a["out"], a["A_log"], a["dt_bias"], ctypes.c_float(a["lb"]), a["init"],
                        a["fin"], a["sdt"], a["cu"], a["nseq"], a["B"], a["T"], a["H"], a["K"],
                        a["V"], a["stream"])


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "out", "A_log", "dt_bias"])
def test_null_pointer_rejected(L, name):
    assert call(**{name: None, "K": 128}) == kda.KDA_ERR_NULL


def test_null_token_pointers_need_empty_tokens(L):
    # T == 0 allows NULL token tensors; this call still fails (bad lower bound), so
    # nothing is launched, but it must not fail on the NULL pointers.
    assert call(q=None, k=None, v=None, g=None, beta=None, out=None, T=0, lb=1.0) == \
        kda.KDA_ERR_VALUE


@pytest.mark.parametrize("K,V", [(64, 128), (128, 64), (256, 256), (0, 128)])
def test_head_size_other_than_128_unsupported(L, K, V):
    assert call(K=K, V=V) == kda.KDA_ERR_UNSUPPORTED


def test_negative_sizes_rejected(L):
    assert call(B=-1) == kda.KDA_ERR_SHAPE
    assert call(T=-5) == kda.KDA_ERR_SHAPE
    assert call(H=-2) == kda.KDA_ERR_SHAPE


def test_cu_seqlens_requires_batch_one(L):
    assert call(cu=P[8], nseq=3, B=2) == kda.KDA_ERR_SHAPE
    assert call(cu=P[8], nseq=0, B=1) == kda.KDA_ERR_SHAPE


def test_state_dtype_rules(L):
    assert call(init=P[9], sdt=kda.KDA_STATE_NONE) == kda.KDA_ERR_DTYPE
    assert call(fin=P[9], sdt=7) == kda.KDA_ERR_DTYPE
    assert call(sdt=5) == kda.KDA_ERR_DTYPE


@pytest.mark.parametrize("lb", [-5.01, 0.5, float("nan"), float("inf")])
def test_lower_bound_range(L, lb):
    assert call(lb=lb, K=128) == kda.KDA_ERR_VALUE


def test_nonfinite_scale(L):
    assert call(scale=float("nan")) == kda.KDA_ERR_VALUE


@pytest.mark.parametrize("name", ["q", "out", "dt_bias"])
def test_misaligned_pointer(L, name):
    assert call(**{name: ctypes.c_void_p(0x10008)}) == kda.KDA_ERR_ALIGN
    assert call(**{name: ctypes.c_void_p(0x10008)}, init=ctypes.c_void_p(0x20004),
                sdt=kda.KDA_STATE_FP32) == kda.KDA_ERR_ALIGN


def test_binding_state_dtype_code():
    import torch
    a32, a16 = torch.zeros(1), torch.zeros(1, dtype=torch.bfloat16)
    assert kda.state_dtype_code(None, None) == kda.KDA_STATE_NONE
    assert kda.state_dtype_code(a32, None) == kda.KDA_STATE_FP32
    assert kda.state_dtype_code(None, a16) == kda.KDA_STATE_BF16
    with pytest.raises(ValueError):
        kda.state_dtype_code(a32, a16)
    with pytest.raises(ValueError):
        kda.state_dtype_code(torch.zeros(1, dtype=torch.float16), None)


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.kda_fwd(x, x, x, x, torch.zeros(1, 4, 2, dtype=torch.bfloat16), 0.1, x,
                    torch.zeros(2), torch.zeros(2, 128), -5.0)


def call_ws(ws=P[10], ws_bytes=1 << 30, **over):
    a = dict(q=P[0], k=P[1], v=P[2], g=P[3], beta=P[4], scale=0.088, out=P[5], A_log=P[6],
             dt_bias=P[7], lb=-5.0, init=None, fin=None, sdt=0, cu=None, nseq=0,
             B=1, T=64, H=2, K=128, V=128, stream=None)
    a.update(over)
    return kda.raw_call_ws(a["q"], a["k"], a["v"], a["g"], a["beta"], ctypes.c_float(a["scale"]),
                           a["out"], a["A_log"], a["dt_bias"], ctypes.c_float(a["lb"]), a["init"],
                           a["fin"], a["sdt"], a["cu"], a["nseq"], a["B"], a["T"], a["H"], a["K"],
                           a["V"], ws, ctypes.c_size_t(ws_bytes), a["stream"])


def test_workspace_size_constant_matches_header():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    m = re.search(r"#define KDA_WORKSPACE_BYTES_PER_UNIT (\d+)", src)
    assert m and int(m.group(1)) == kda.WORKSPACE_BYTES_PER_UNIT
    assert kda.workspace_bytes(3, 4) == 12 * kda.WORKSPACE_BYTES_PER_UNIT


def test_ws_entry_point_validates_workspace(L):
    need = 1 * 2 * kda.WORKSPACE_BYTES_PER_UNIT
    # every case below still fails validation, so nothing is launched on the fake pointers
    assert call_ws(ws=None, ws_bytes=need) == kda.KDA_ERR_NULL
    assert call_ws(ws=ctypes.c_void_p(0x10008), ws_bytes=need) == kda.KDA_ERR_ALIGN
    assert call_ws(ws_bytes=need - 16) == kda.KDA_ERR_VALUE
    # the ordinary argument checks come first
    assert call_ws(K=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_ws(lb=1.0) == kda.KDA_ERR_VALUE
    # no work: a NULL workspace of size 0 is accepted without touching the device
    assert call_ws(ws=None, ws_bytes=0, q=None, k=None, v=None, g=None, beta=None, out=None,
                   B=0) == kda.KDA_OK


def call_unbounded(**over):
    a = dict(q=P[0], k=P[1], v=P[2], g=P[3], beta=P[4], scale=0.088, out=P[5], A_log=P[6],
             dt_bias=P[7], init=None, fin=None, sdt=0, cu=None, nseq=0,
             B=1, T=64, H=2, K=128, V=128, stream=None)
    a.update(over)
    return kda.lib().kda_fwd_unbounded(a["q"], a["k"], a["v"], a["g"], a["beta"],
                                       ctypes.c_float(a["scale"]), a["out"], a["A_log"],
                                       a["dt_bias"], a["init"], a["fin"], a["sdt"], a["cu"],
                                       a["nseq"], a["B"], a["T"], a["H"], a["K"], a["V"],
                                       a["stream"])


def test_unbounded_gate_entry_point_validates(L):
    # every case fails validation (nothing launched on the fake pointers), except the
    # last, which has no work
    assert call_unbounded(K=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_unbounded(q=None) == kda.KDA_ERR_NULL
    assert call_unbounded(out=ctypes.c_void_p(0x10008)) == kda.KDA_ERR_ALIGN
    assert call_unbounded(scale=float("inf")) == kda.KDA_ERR_VALUE
    assert call_unbounded(init=P[9], sdt=kda.KDA_STATE_NONE) == kda.KDA_ERR_DTYPE
    assert call_unbounded(cu=P[8], nseq=2, B=3) == kda.KDA_ERR_SHAPE
    assert call_unbounded(q=None, k=None, v=None, g=None, beta=None, out=None, B=0) == kda.KDA_OK


def test_too_many_units_rejected(L):
    # N * H above 2^26 - 1 would overflow the widest grid; rejected before any launch
    assert call(B=1 << 20, H=128, T=1) == kda.KDA_ERR_SHAPE
    assert call(B=1 << 40, H=1 << 30, T=1) == kda.KDA_ERR_SHAPE   # no int64 overflow either
    assert call_unbounded(B=1 << 20, H=128, T=1) == kda.KDA_ERR_SHAPE


def test_workspace_size_query(L):
    assert L.kda_workspace_size(3, 5) == 3 * 5 * kda.WORKSPACE_BYTES_PER_UNIT == kda.workspace_bytes(3, 5)
    assert L.kda_workspace_size(0, 5) == 0 and L.kda_workspace_size(3, 0) == 0
    assert L.kda_workspace_size(-1, 5) == 0 and L.kda_workspace_size(3, -2) == 0
    assert L.kda_workspace_size(1 << 40, 1 << 30) == 0   # does not fit in size_t
    # the pool-sized workspace: 0 for sizes out of range, and (it queries the device's SM
    # count) without a device; with one, at least the cluster kernel's size
    assert L.kda_workspace_size_pool(0, 5) == 0 and L.kda_workspace_size_pool(-1, 5) == 0
    assert L.kda_workspace_size_pool(3, 1 << 40) == 0
    n = L.kda_workspace_size_pool(3, 5)
    assert n == 0 or n >= L.kda_workspace_size(3, 5)


def test_static_entry_point_rejects_calls_above_its_limit(L):
    # the unit limit is checked after the ordinary validation and before any device call
    def call_static(**over):
        a = dict(q=P[0], k=P[1], v=P[2], g=P[3], beta=P[4], out=P[5], A_log=P[6], dt_bias=P[7],
                 B=1, T=64, H=kda.STATIC_MAX_UNITS + 1, K=128)
        a.update(over)
        return L.kda_fwd_static(a["q"], a["k"], a["v"], a["g"], a["beta"], ctypes.c_float(0.088),
                                a["out"], a["A_log"], a["dt_bias"], ctypes.c_float(-5.0), None,
                                None, 0, None, 0, a["B"], a["T"], a["H"], a["K"], 128, None)
    assert call_static() == kda.KDA_ERR_LIMIT
    assert call_static(B=3, H=kda.STATIC_MAX_UNITS // 2) == kda.KDA_ERR_LIMIT
    assert call_static(K=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_static(q=None, k=None, v=None, g=None, beta=None, out=None, B=0) == kda.KDA_OK
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    m = re.search(r"#define KDA_STATIC_MAX_UNITS (\d+)", src)
    assert m and int(m.group(1)) == kda.STATIC_MAX_UNITS
