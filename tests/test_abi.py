"""The C-ABI library on the CPU: it loads, exports every entry point that
include/ozk.h declares, and its host-side logic (moduli, bit budget, slice
padding, workspace size, status text) agrees with the oracle and with itself.
No compute call is made here (no GPU)."""
import ctypes
import os
import re

import pytest

import oracle
from fp64_gemm_emulation_exponent_gb300 import build as ozk_build
from fp64_gemm_emulation_exponent_gb300 import ozk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ozk.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    ozk_build.build()
    yield


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ozk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ["ozk_dgemm", "ozk_dgemm_ws", "ozk_workspace_size", "ozk_stream_status",
                 "ozk_status_string", "ozk_scale", "ozk_quantize_a", "ozk_quantize_b",
                 "ozk_residue_gemm", "ozk_crt_combine", "ozk_crt_lift"]:
        assert must in names


def test_library_exports_every_declared_symbol():
    L = ozk.lib()
    missing = [name for name in declared_functions() if not hasattr(L, name)]
    assert not missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) == set(ozk.SIGNATURES)


def test_moduli_match_the_oracle():
    assert ozk.ozk_moduli(20) == [int(p) for p in oracle.moduli(20)]


def test_beta_matches_the_oracle():
    for n in range(2, 21):
        for K in [1, 2, 3, 63, 64, 65, 255, 256, 512, 1000, 1024, 4096, 8192, 65536, 131071, 131072, 10**6, 4194304]:
            try:
                want = oracle.beta(K, n)
            except oracle.OracleError:
                want = -ozk.OZK_ERR_UNSUPPORTED
            assert ozk.ozk_beta(K, n) == want, (K, n)


def test_moduli_for_bits_is_the_smallest_count_reaching_the_target():
    # against the oracle's own beta: the chosen count reaches the target and one fewer does not
    for K in [1, 64, 1000, 4096, 8192, 65536, 131072, 10**6]:
        betas = {}
        for n in range(2, 21):
            try:
                betas[n] = oracle.beta(K, n)
            except oracle.OracleError:
                betas[n] = 0
        for target in [1, 8, 20, 26, 30, 34, 40, 46, 48, 50, 53, 60, 72, 80]:
            got = ozk.ozk_moduli_for_bits(K, target)
            reach = [n for n in range(2, 21) if betas[n] >= target]
            if not reach:
                assert got == -ozk.OZK_ERR_UNSUPPORTED, (K, target)
            else:
                assert got == reach[0], (K, target)
    assert ozk.ozk_moduli_for_bits(4096, 0) == -ozk.OZK_ERR_INVALID_ARG


def test_gamma_matches_the_oracle():
    for n in range(2, 21):
        for K in [1, 2, 63, 64, 1000, 4096, 65536, 131072, 10**6, 4194304]:
            try:
                want = oracle.gamma(K, n)
            except oracle.OracleError:
                want = -ozk.OZK_ERR_UNSUPPORTED
            assert ozk.ozk_gamma(K, n) == want, (K, n)


def test_workspace_layout_regions_fit_and_do_not_overlap():
    for (M, N, K, n) in [(1, 1, 1, 2), (300, 257, 700, 14), (2048, 1024, 2100, 14), (300, 257, 9000, 13),
                         (300, 257, 33000, 13), (96, 80, 140000, 14), (8192, 8192, 512, 20)]:
        info = ozk.ozk_workspace_layout(M, N, K, n)
        assert info.total_bytes == ozk.ozk_workspace_size(M, N, K, n)
        assert info.kpad == ozk.ozk_kpad(K)
        esize = {0: 1, 1: 4, 2: 2}[info.planes_kind]
        planes = {0: n, 1: n * info.splits, 2: (n + 1) // 2}[info.planes_kind]
        regions = [(info.maxima_offset, 2 * 8 * (M + N)), (info.s_offset, 4 * M), (info.t_offset, 4 * N),
                   (info.a_slices_offset, 2 * ((n - 1) * info.a_plane + M * info.kpad)),
                   (info.b_slices_offset, 2 * ((n - 1) * info.b_plane + N * info.kpad)),
                   (info.planes_offset, esize * ((planes - 1) * info.planes_plane + M * info.planes_ld))]
        end = 0
        for off, size in regions:
            assert off >= end and off % 256 == 0
            end = off + size
        assert end <= info.total_bytes
        assert info.a_plane >= M * info.kpad and info.b_plane >= N * info.kpad
        assert info.planes_ld >= N and info.planes_plane >= M * info.planes_ld


def test_split_count_keeps_its_constraints():
    """The K split count of ozk_dgemm's residue GEMM: at least the shares K
    beyond one int32-exact sum needs, at most 64, every share at least 2048
    of K (the CTA-pair kernel's minimum) when K is split, int32 partial sums
    exactly when it is split, and none where whole-K units already fill the
    GPU (square products)."""
    shapes = [(M, N, K, n) for (M, N) in [(64, 64), (256, 256), (512, 512), (600, 520), (1024, 1024), (2048, 72),
                                          (4096, 4096)]
              for K in [512, 2048, 4096, 33000, 65536, 131072, 300000, 1 << 20] for n in [2, 8, 14, 20]]
    for (M, N, K, n) in shapes:
        if ozk.ozk_beta(K, n) < 1:
            continue
        info = ozk.ozk_workspace_layout(M, N, K, n)
        kpad, sp = info.kpad, info.splits
        assert -(-kpad // ozk.OZK_SPLIT_MAX_K) <= sp <= 64, (M, N, K, n, sp)
        assert (info.planes_kind == 1) == (sp > 1), (M, N, K, n)
        if sp > 1:
            assert kpad // 64 // sp >= 2048 // 64, (M, N, K, n, sp)
            assert -(-(kpad // 64) // sp) * 64 <= ozk.OZK_SPLIT_MAX_K
    for (M, N, K) in [(4096, 4096, 4096), (8192, 8192, 8192), (8192, 8192, 512), (2048, 2048, 32768)]:
        assert ozk.ozk_workspace_layout(M, N, K, 14).splits == 1
    # the choices measured best on 512^2 x 65536: unsplit where 56 or 68 units
    # already keep HBM busy, split where 80 units would leave a second wave of 4
    assert [ozk.ozk_workspace_layout(512, 512, 65536, n).splits for n in (14, 17, 20)] == [1, 1, 4]


def test_quantiser_residue_division_is_exact_below_two_to_the_20():
    """The quantiser forms each residue from x, the bytes of the offset
    integer (up to twelve) against 2^(8b) mod p plus an offset below 2p:
    x < 12 * 255 * 254 + 2p < 2^20.  It divides by a multiply-high with
    ceil(2^32 / p); that quotient is floor(x / p) for every such x and every
    odd modulus."""
    import numpy as np

    assert 12 * 255 * 254 + 2 * 256 < 1 << 20
    x = np.arange(1 << 20, dtype=np.uint64)
    for p in (int(v) for v in oracle.moduli(ozk.OZK_MAX_MODULI)):
        if p == 256:
            continue
        m32 = np.uint64(((1 << 32) + p - 1) // p)
        assert np.array_equal((x * m32) >> np.uint64(32), x // np.uint64(p)), p


def test_kpad():
    assert [ozk.ozk_kpad(k) for k in [0, 1, 63, 64, 65, 128, 131071]] == [0, 64, 64, 64, 128, 128, 131072]


def test_workspace_size():
    assert ozk.ozk_workspace_size(0, 10, 10, 14) == 0
    assert ozk.ozk_workspace_size(10, 10, 0, 14) == 0
    assert ozk.ozk_workspace_size(10, 10, 10, 1) == 0
    assert ozk.ozk_workspace_size(10, 10, ozk.OZK_MAX_K + 1, 14) == 0
    # K beyond one int32-exact sum: int32 partial planes of at least ceil(kpad / OZK_SPLIT_MAX_K) splits
    for K in (131072, 10**6, ozk.OZK_MAX_K):
        kpad = ozk.ozk_kpad(K)
        min_splits = -(-kpad // ozk.OZK_SPLIT_MAX_K)
        assert ozk.ozk_workspace_size(10, 10, K, 14) >= 2 * 14 * 20 * kpad + 4 * min_splits * 14 * 10 * 12
    for (M, N, K, n) in [(1, 1, 1, 2), (256, 256, 256, 14), (4096, 4096, 4096, 14), (8192, 8192, 512, 20),
                         (512, 512, 65536, 20)]:
        ws = ozk.ozk_workspace_size(M, N, K, n)
        kpad = ozk.ozk_kpad(K)
        slices = 2 * n * (M + N) * kpad
        assert ws >= slices + n * M * N
        assert ws % 256 == 0
    # grows with every dimension
    base = ozk.ozk_workspace_size(300, 300, 300, 14)
    assert ozk.ozk_workspace_size(301, 300, 300, 14) > base
    assert ozk.ozk_workspace_size(300, 300, 400, 14) > base
    assert ozk.ozk_workspace_size(300, 300, 300, 15) > base


def test_status_strings():
    for code in range(0, 7):
        assert ozk.status_string(code)
    assert ozk.status_string(99) == "unknown status"


def test_argument_errors_come_back_before_any_cuda_call():
    """Every GEMM entry point checks its arguments on the host and returns
    the error before touching CUDA, so these calls run on a machine without a
    GPU; an empty C is a no-op that succeeds there too."""
    L = ozk.lib()
    p = ctypes.c_void_p
    bufs = [(ctypes.c_double * 64)() for _ in range(3)]
    a, b, c = (ctypes.cast(x, p) for x in bufs)
    for name in ("ozk_dgemm", "ozk_dgemm_host", "ozk_dgemm_host_async"):
        f = getattr(L, name)
        assert f(-1, 2, 2, a, 2, b, 2, c, 2, 14, None) == ozk.OZK_ERR_INVALID_ARG
        assert f(2, 2, 2, a, 2, b, 2, c, 2, 1, None) == ozk.OZK_ERR_UNSUPPORTED        # n_moduli < 2
        assert f(2, 2, 2, a, 2, b, 2, c, 2, 21, None) == ozk.OZK_ERR_UNSUPPORTED       # n_moduli > 20
        assert f(2, 2, ozk.OZK_MAX_K + 1, a, ozk.OZK_MAX_K + 1, b, 2, c, 2, 14, None) == ozk.OZK_ERR_UNSUPPORTED
        assert f(2, 2, 2, None, 2, b, 2, c, 2, 14, None) == ozk.OZK_ERR_INVALID_ARG    # null A
        assert f(2, 2, 2, a, 1, b, 2, c, 2, 14, None) == ozk.OZK_ERR_INVALID_ARG       # lda < K
        assert f(2, 2, 2, a, 2, b, 2, c, 1, 14, None) == ozk.OZK_ERR_INVALID_ARG       # ldc < N
        assert f(2, 2, 2, a, 2, b, 2, a, 2, 14, None) == ozk.OZK_ERR_INVALID_ARG       # C overlaps A
        assert f(2, 2, 60000, a, 60000, b, 2, c, 2, 2, None) == ozk.OZK_ERR_UNSUPPORTED  # beta < 1
        assert f(0, 5, 3, None, 3, None, 5, None, 5, 14, None) == ozk.OZK_OK           # empty C
    assert L.ozk_dgemm_ws(2, 2, 2, a, 2, b, 2, c, 2, 1, None, 0, None) == ozk.OZK_ERR_UNSUPPORTED
    assert L.ozk_dgemm_bits(2, 2, 2, a, 2, b, 2, c, 2, 0, None) == ozk.OZK_ERR_INVALID_ARG   # target < 1
    assert L.ozk_dgemm_bits(2, 2, 2, a, 2, b, 2, c, 2, 200, None) == ozk.OZK_ERR_UNSUPPORTED
    # the failure-path test hook: the single-CTA kernel only, a k-block that
    # exists and a time limit of 1 us .. 1 s
    w = L.ozk_residue_gemm_withheld
    assert w(2, 2, 2048, a, b, 2, c, 16, 0, 1000, None) == ozk.OZK_ERR_INVALID_ARG
    assert w(2, 2, 64, a, b, 2, c, 16, 1, 1000, None) == ozk.OZK_ERR_INVALID_ARG
    assert w(2, 2, 64, a, b, 2, c, 16, 0, 0, None) == ozk.OZK_ERR_INVALID_ARG
    assert w(2, 2, 64, a, b, 2, c, 16, 0, 2000000, None) == ozk.OZK_ERR_INVALID_ARG
    assert w(2, 2, 64, a, b, 1, c, 16, 0, 1000, None) == ozk.OZK_ERR_UNSUPPORTED
