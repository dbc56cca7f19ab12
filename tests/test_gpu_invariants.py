"""Properties of the operators checked directly on the CUDA library, and its
device-side argument checks and bounded-wait failure path."""
import ctypes

import numpy as np
import pytest

from inputs import grid_coords
from tests.gpu_helpers import TOL_ACCURATE, dev, host_complex, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()


def _fhd(kx, ky, kz, D, x, y, z, mode=0):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    f = lambda a: dev(np.asarray(a, dtype=np.float32))
    rr, ri = fhd.fhd_compute(f(kx), f(ky), f(kz), f(D.real), f(D.imag), f(x), f(y), f(z), mode=mode)
    torch.cuda.synchronize()
    return host_complex(rr, ri)


@pytest.mark.parametrize("mode", [0, 1])
def test_k0_gives_D0(mode):
    x, y, z = (np.random.default_rng(1).uniform(-0.5, 0.5, 5000) for _ in range(3))
    D = np.array([0.75 - 1.25j])
    got = _fhd([0.0], [0.0], [0.0], D, x, y, z, mode)
    assert np.max(np.abs(got - D[0])) <= 1e-6


@pytest.mark.parametrize("mode", [0, 1])
def test_hermitian_data_gives_real_image(mode):
    rng = np.random.default_rng(2)
    h = rng.uniform(-30, 30, size=(1500, 3)).astype(np.float32)
    k = np.concatenate([h, -h])
    Dh = rng.standard_normal(1500) + 1j * rng.standard_normal(1500)
    D = np.concatenate([Dh, np.conj(Dh)]).astype(np.complex64)
    x, y, z = grid_coords(16, 16, 16)
    got = _fhd(k[:, 0], k[:, 1], k[:, 2], D, x, y, z, mode)
    assert np.linalg.norm(got.imag) <= (1e-5 if mode == 0 else 1e-3) * np.linalg.norm(got.real)


@pytest.mark.parametrize("mode", [0, 1])
def test_cartesian_is_inverse_fft(mode):
    """All integer k in [-n/2, n/2)^3 on the n^3 grid: F^H D = n^3 ifftn(D (-1)^(sum k))."""
    n = 16
    x, y, z = grid_coords(n, n, n)
    ks = np.arange(n) - n // 2
    KZ, KY, KX = np.meshgrid(ks, ks, ks, indexing="ij")
    rng = np.random.default_rng(3)
    D = (rng.standard_normal(KX.size) + 1j * rng.standard_normal(KX.size)).astype(np.complex64)
    A = np.zeros((n, n, n), dtype=np.complex128)
    A[KZ.ravel() % n, KY.ravel() % n, KX.ravel() % n] = D.astype(np.complex128) * (-1.0) ** (KX + KY + KZ).ravel()
    ref = n ** 3 * np.fft.ifftn(A).ravel()
    got = _fhd(KX.ravel(), KY.ravel(), KZ.ravel(), D, x, y, z, mode)
    assert rel_l2(got, ref) <= (TOL_ACCURATE if mode == 0 else 1e-3)


def test_adjoint_identity_on_gpu():
    """<F rho, D> = <rho, F^H D> using only the CUDA operators."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    rng = np.random.default_rng(4)
    N, M = 6000, 3000
    f = lambda a: dev(np.asarray(a, dtype=np.float32))
    x, y, z = (f(rng.uniform(-0.5, 0.5, N)) for _ in range(3))
    kx, ky, kz = (f(rng.uniform(-25, 25, M)) for _ in range(3))
    rho = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    D = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    Fr, Fi = fhd.fwd_compute(x, y, z, f(rho.real), f(rho.imag), kx, ky, kz)
    Hr, Hi = fhd.fhd_compute(kx, ky, kz, f(D.real), f(D.imag), x, y, z)
    torch.cuda.synchronize()
    rho32 = rho.astype(np.complex64).astype(np.complex128)
    D32 = D.astype(np.complex64).astype(np.complex128)
    lhs = np.vdot(host_complex(Fr, Fi), D32)
    rhs = np.vdot(rho32, host_complex(Hr, Hi))
    assert abs(lhs - rhs) <= 1e-5 * np.sqrt(N * M)


# ------------------------------------------------------------ device-side argument checks

def _raw(lib, M, kp, N, xp, out, ws, wsb):
    return lib.fhd_compute(M, *kp, N, *xp, *out, 0, ws, wsb, None)


# The pointer checks run through fhd_test_check_array, which launches nothing:
# a pointer the check should reject is never handed to a kernel here.

def test_check_accepts_device_memory():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    lib = fhd.load()
    d = torch.zeros(1000, device="cuda")
    assert lib.fhd_test_check_array(d.data_ptr(), 4000, 0) == 0
    assert lib.fhd_test_check_array(d.data_ptr() + 2, 400, 0) == 2


def test_check_rejects_host_memory():
    import non_cartesian_mri_gather_gb300 as fhd

    lib = fhd.load()
    host = np.zeros(64, dtype=np.float32)
    assert lib.fhd_test_check_array(host.ctypes.data, 256, 0) == 1


def test_check_rejects_past_allocation_end():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    lib = fhd.load()
    torch.cuda.empty_cache()
    big = torch.zeros(8 << 20, device="cuda")  # 32 MiB
    tail = big[-100:]
    assert lib.fhd_test_check_array(tail.data_ptr(), 400, 0) == 0
    assert lib.fhd_test_check_array(tail.data_ptr(), 4000, 0) == 7


def test_rejects_small_workspace():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    lib = fhd.load()
    d = torch.zeros(500, device="cuda")
    outs = [torch.empty(500, device="cuda") for _ in range(2)]
    need = fhd.fhd_workspace_bytes(fhd.OP_FHD, 500, 500)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = _raw(lib, 500, [d.data_ptr()] * 5, 500, [d.data_ptr()] * 3, [o.data_ptr() for o in outs], ws.data_ptr(),
              need - 256)
    assert st == 4


# ------------------------------------------------------------ bounded-wait failure path

def test_timeout_is_reported_and_context_survives():
    """The producer skips one tile's copy: the consumers' bounded wait expires,
    the status word reports FHD_ERR_TIMEOUT, and the next call works."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    from inputs import random_problem

    lib = fhd.load()
    p = random_problem(5000, 2000, kmax=16.0, seed=9)
    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
    out = [torch.empty(p.N, device="cuda") for _ in range(2)]
    ws = fhd.Workspace(fhd.OP_FHD, p.N, p.M)
    stream = torch.cuda.current_stream().cuda_stream
    args = (p.M, t["kx"].data_ptr(), t["ky"].data_ptr(), t["kz"].data_ptr(), t["Dr"].data_ptr(), t["Di"].data_ptr(),
            p.N, t["x"].data_ptr(), t["y"].data_ptr(), t["z"].data_ptr(), out[0].data_ptr(), out[1].data_ptr(), 0,
            ws.ptr, ws.nbytes, stream)
    assert lib.fhd_test_compute_skip_tile(*args, 3) == 0
    assert fhd.fhd_workspace_status(ws) == 6
    # the context is still usable and the status word is cleared by the next call
    assert lib.fhd_test_compute_skip_tile(*args, -1) == 0
    assert fhd.fhd_workspace_status(ws) == 0
    torch.cuda.synchronize()
    import oracle

    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    assert rel_l2(host_complex(*out), ref) <= TOL_ACCURATE


# ------------------------------------------------------------ profiling entry point and launch shape

@pytest.mark.parametrize("N,M", [(1024, 2048), (65536, 4096)])
@pytest.mark.parametrize("mode", [0, 1])
def test_profiled_call_matches_and_times_the_gather(N, M, mode):
    """fhd_compute_profiled gives fhd_compute's result bit for bit (split path
    for the small size, persistent gather for the large one) and its two
    events bracket a positive device time shorter than the whole call's."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    from inputs import random_problem

    p = random_problem(N, M, kmax=16.0, seed=N + M)
    t = {k: dev(getattr(p, k)) for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")}
    ws = fhd.Workspace(fhd.OP_FHD, N, M)
    args = [t[k] for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")]
    a = fhd.fhd_compute(*args, mode=mode, workspace=ws)
    out = (torch.empty(N, device="cuda"), torch.empty(N, device="cuda"))
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    fhd.fhd_compute_profiled(*args, out[0], out[1], mode, ws, g0, g1)
    c1.record()
    torch.cuda.synchronize()
    assert np.array_equal(host_complex(*a), host_complex(*out))
    gather_ms, call_ms = g0.elapsed_time(g1), c0.elapsed_time(c1)
    assert 0.0 < gather_ms <= call_ms


def test_launch_shape():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for mode in (0, 1, 2, 3):
        shape = fhd.fhd_launch_shape(0, mode)
        assert shape["ctas"] == sms
        assert (shape["threads"], shape["targets_per_thread"], shape["tile_sources"], shape["stages"]) == (256, 32, 256, 5)
    lib = fhd.load()
    vals = [ctypes.c_int(0) for _ in range(5)]
    assert lib.fhd_launch_shape(0, 4, *(ctypes.addressof(v) for v in vals)) == 1  # unknown mode bit


def test_concurrent_calls_on_two_streams():
    """Two calls in flight at once on different streams, each with its own
    workspace (the header's rule), give their sequential results bit for bit:
    a persistent gather and a split gather, and an F^H F rho beside an F^H D."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    from inputs import random_problem

    big = random_problem(65536, 4096, kmax=16.0, seed=51, coords="grid")
    small = random_problem(1500, 3000, kmax=16.0, seed=52)
    fhf = random_problem(20000, 3000, kmax=12.0, seed=53, op="fhf")
    tb = {k: dev(getattr(big, k)) for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")}
    ts = {k: dev(getattr(small, k)) for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")}
    tf = {k: dev(getattr(fhf, k)) for k in ("x", "y", "z", "rho_r", "rho_i", "kx", "ky", "kz")}
    ab = [tb[k] for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")]
    as_ = [ts[k] for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")]
    af = [tf[k] for k in ("x", "y", "z", "rho_r", "rho_i", "kx", "ky", "kz")]
    wb = fhd.Workspace(fhd.OP_FHD, big.N, big.M)
    ws_ = fhd.Workspace(fhd.OP_FHD, small.N, small.M)
    wf = fhd.Workspace(fhd.OP_FHF, fhf.N, fhf.M)
    ref_b = host_complex(*fhd.fhd_compute(*ab, mode=1, workspace=wb))
    ref_s = host_complex(*fhd.fhd_compute(*as_, mode=1, workspace=ws_))
    ref_f = host_complex(*fhd.fhfrho_apply(*af, mode=1, workspace=wf))
    torch.cuda.synchronize()
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        ob = fhd.fhd_compute(*ab, mode=1, workspace=wb, stream=s1)
        os_ = fhd.fhd_compute(*as_, mode=1, workspace=ws_, stream=s2)
        of = fhd.fhfrho_apply(*af, mode=1, workspace=wf, stream=s3)
        torch.cuda.synchronize()
        assert np.array_equal(host_complex(*ob), ref_b)
        assert np.array_equal(host_complex(*os_), ref_s)
        assert np.array_equal(host_complex(*of), ref_f)
    for w, s in ((wb, s1), (ws_, s2), (wf, s3)):
        assert fhd.fhd_workspace_status(w, s) == 0


def test_fma2_rate_probe():
    """The packed-FMA probe reports a rate between a third of and just above
    the nominal FP32 lane peak (128 lanes per SM per clock, at most about
    2.1 GHz), and rejects a null output pointer."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    rate = ctypes.c_double(0.0)
    assert fhd.load().fhd_test_fma2_rate(0, ctypes.byref(rate)) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nominal_max = sms * 128 * 2.1e9
    assert nominal_max / 3 < rate.value < 1.05 * nominal_max, rate.value
    assert fhd.load().fhd_test_fma2_rate(0, None) == 1  # FHD_ERR_INVALID_VALUE
