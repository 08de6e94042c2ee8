"""tcgen05 building blocks on the GPU: single MMAs through the shared-memory
descriptor encodings (K-major and MN-major 128B-swizzled tiles, M = 128, the N
and K extents the KDA kernel uses) against torch.matmul, plus a TMEM store/load
round trip."""
import ctypes
import glob
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
PROBE_SRC = os.path.join(HERE, "csrc", "tc_probe.cu")
PROBE_OUT = os.path.join(HERE, "csrc", "libkda_probe.so")


def build_probe() -> str:
    """Builds the probe library (tests/csrc/libkda_probe.so) with the product's flags."""
    from gated_delta_rule_52_gb300 import build
    hdrs = glob.glob(os.path.join(build.CSRC, "*.cuh"))
    if os.path.exists(PROBE_OUT) and all(os.path.getmtime(f) <= os.path.getmtime(PROBE_OUT)
                                         for f in [PROBE_SRC, *hdrs]):
        return PROBE_OUT
    tmp = PROBE_OUT + f".tmp{os.getpid()}"
    cmd = [build.nvcc(), *build.ARCH, *build.FLAGS, "-shared", "-o", tmp, PROBE_SRC, "-lcuda"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    os.replace(tmp, PROBE_OUT)
    return PROBE_OUT


@pytest.fixture(scope="module")
def probe():
    L = ctypes.CDLL(build_probe())
    L.kda_probe_mma.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 2
    L.kda_probe_mma.restype = ctypes.c_int
    return L


CASES = [(N, K, a, b, f) for (N, K) in [(64, 64), (64, 128), (128, 128), (160, 128), (192, 64),
                                        (256, 64)]
         for a in (0, 1) for b in (0, 1) for f in (0, 1) if not (b and N % 64)]


@pytest.mark.parametrize("N,K,a_mn,b_mn,fp16", CASES)
def test_mma_layouts(probe, N, K, a_mn, b_mn, fp16):
    g = torch.Generator(device="cpu").manual_seed(N * 1000 + K * 10 + 2 * a_mn + b_mn)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(K, N, generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.kda_probe_mma(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, fp16,
                             st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0, f"probe status {st.item()}"
    # bf16 inputs convert exactly to fp16 at these magnitudes, so both kinds match
    ref = A.float() @ B.float()
    torch.testing.assert_close(D, ref, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("T,H,h,t0,c0", [(256, 4, 1, 0, 0), (256, 4, 3, 37, 64), (100, 2, 0, 70, 0),
                                         (300, 64, 63, 256, 64)])
def test_tma_3d_swizzled_load(probe, T, H, h, t0, c0):
    probe.kda_probe_tma.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p]
    probe.kda_probe_tma.restype = ctypes.c_int
    g = torch.Generator(device="cpu").manual_seed(T + H + h + t0 + c0)
    src = torch.randn(T, H, 128, generator=g).to(torch.bfloat16).cuda()
    out = torch.full((64, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.kda_probe_tma(src.data_ptr(), T, H, h, t0, c0, out.data_ptr(), st.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    n = max(0, min(64, T - t0))
    ref[:n] = src[t0:t0 + n, h, c0:c0 + 64]
    assert torch.equal(out, ref)


def test_bounded_wait_gives_up_and_the_context_stays_usable(probe):
    # The wait every libkda kernel uses, on a barrier that nothing arrives on: it must
    # give up after its limit (the kernels then set the device error word and unwind).
    probe.kda_probe_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    probe.kda_probe_wait.restype = ctypes.c_int
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert probe.kda_probe_wait(5_000_000, 0, out.data_ptr(), s) == 0   # 5 ms, never arrived
    torch.cuda.synchronize()
    status, ns = out.tolist()
    assert status == 2 and 5_000_000 <= ns < 500_000_000, (status, ns)
    assert probe.kda_probe_wait(5_000_000, 1, out.data_ptr(), s) == 0   # completed barrier
    torch.cuda.synchronize()
    status, ns = out.tolist()
    assert status == 1 and ns < 5_000_000, (status, ns)
    # the context still runs work afterwards
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1024 * 1023 / 2
