"""hs_gemm_bf16 and hs_gemm_bf16_swiglu (the hybrid stack's projections and MLPs) against a plain fp32 PyTorch product of the same
bf16 operands: C = A B^T (+ R) with C and R in bf16 or fp32, ragged M, N = 128 odd multiples (a last
256-wide column block half out of range), R aliasing C; and batch invariance: a row's bits do not depend on
how many rows share the launch (Flide section 3.5)."""
import pytest
import torch

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import _lib  # noqa: E402
from hybrid_serving_gb300.stack import gemm  # noqa: E402


def _ref(A, B, R=None):
    out = A.float() @ B.float().t()
    return out + R.float() if R is not None else out


@pytest.mark.parametrize("M, N, K", [(1, 128, 64), (300, 384, 128), (1000, 2048, 2048), (4099, 6272, 256),
                                     (257, 512, 4096)])
@pytest.mark.parametrize("cdt, res", [(torch.bfloat16, False), (torch.bfloat16, True), (torch.float32, True),
                                      (torch.float32, False)])
def test_gemm_matches_fp32_product(M, N, K, cdt, res):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    C = torch.randn(M, N, device="cuda", generator=g).to(cdt)  # the residual, added in place
    R0 = C.clone() if res else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gemm(A, B, C, M, R=C if res else None, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = _ref(A, B, R0)
    err = float((C.float() - want).abs().max())
    # fp32 accumulation in another order, then the output's own rounding (bf16: 2^-9 relative)
    scale = float(want.abs().max())
    bar = (2.0 ** -8 if cdt == torch.bfloat16 else 1e-5) * scale + 1e-5 * K ** 0.5
    print(f"[margin] gemm {M}x{N}x{K} {str(cdt)[6:]} res={res}: max-abs {err:.3e} (bar {bar:.2e})")
    assert err <= bar


def test_gemm_rows_do_not_depend_on_m():
    g = torch.Generator(device="cuda").manual_seed(5)
    K, N = 512, 640
    A = torch.randn(3000, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    big = torch.empty(3000, N, device="cuda", dtype=torch.bfloat16)
    gemm(A, B, big, 3000, status=st)
    for m0, m in [(0, 1), (0, 129), (1000, 77), (2871, 129)]:
        small = torch.empty(m, N, device="cuda", dtype=torch.bfloat16)
        gemm(A[m0:m0 + m], B, small, m, status=st)
        torch.cuda.synchronize()
        assert torch.equal(small, big[m0:m0 + m]), (m0, m)
    assert int(st.item()) == 0


def test_gemm_refuses_bad_shapes():
    A = torch.zeros(8, 64, device="cuda", dtype=torch.bfloat16)
    B = torch.zeros(100, 64, device="cuda", dtype=torch.bfloat16)
    C = torch.zeros(8, 100, device="cuda", dtype=torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.HsError) as e:
        gemm(A, B, C, 8, status=st)
    assert e.value.code == _lib.HS_EUNSUPPORTED


@pytest.mark.parametrize("M, F, K", [(1, 128, 64), (300, 384, 128), (1000, 2048, 2048), (257, 512, 4096)])
def test_gemm_swiglu_matches_fp32(M, F, K):
    """hs_gemm_bf16_swiglu against silu(A Bg^T) * (A Bu^T) in fp32 from the same bf16 operands (B given in
    the interleaved row order), and against the unfused path's bits where both round once: C within the
    output's bf16 rounding plus the fp32 products' reordering."""
    from hybrid_serving_gb300.stack import gemm_swiglu, interleave_gate_up
    g = torch.Generator(device="cuda").manual_seed(M * 11 + F + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    Bgu = (torch.randn(2 * F, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    B_il = torch.from_numpy(interleave_gate_up(Bgu.float().cpu().numpy())).to("cuda").to(torch.bfloat16)
    C = torch.full((M, F), float("nan"), device="cuda", dtype=torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gemm_swiglu(A, B_il, C, M, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    gu = A.float() @ Bgu.float().t()
    gt, up = gu[:, :F], gu[:, F:]
    want = gt * torch.sigmoid(gt) * up
    err = float((C.float() - want).abs().max())
    # the products' fp32 reordering (relative ~1e-6 of |g|, |u|) through silu(g) * u, then bf16 rounding
    scale = float(want.abs().max())
    bar = 2.0 ** -8 * scale + 1e-5 * K ** 0.5 * float(gu.abs().max())
    print(f"[margin] gemm swiglu {M}x{F}x{K}: max-abs {err:.3e} (bar {bar:.2e})")
    assert err <= bar


def test_gemm_swiglu_rows_do_not_depend_on_m():
    from hybrid_serving_gb300.stack import gemm_swiglu
    g = torch.Generator(device="cuda").manual_seed(9)
    K, F = 512, 384
    A = torch.randn(3000, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(2 * F, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    big = torch.empty(3000, F, device="cuda", dtype=torch.bfloat16)
    gemm_swiglu(A, B, big, 3000, status=st)
    for m0, m in [(0, 1), (0, 129), (1000, 77), (2871, 129)]:
        small = torch.empty(m, F, device="cuda", dtype=torch.bfloat16)
        gemm_swiglu(A[m0:m0 + m], B, small, m, status=st)
        torch.cuda.synchronize()
        assert torch.equal(small, big[m0:m0 + m]), (m0, m)
    assert int(st.item()) == 0


def test_gemm_swiglu_refuses_bad_shapes():
    from hybrid_serving_gb300.stack import gemm_swiglu
    A = torch.zeros(8, 64, device="cuda", dtype=torch.bfloat16)
    B = torch.zeros(384, 64, device="cuda", dtype=torch.bfloat16)  # N2 not a multiple of 256
    C = torch.zeros(8, 192, device="cuda", dtype=torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.HsError) as e:
        gemm_swiglu(A, B, C, 8, status=st)
    assert e.value.code == _lib.HS_EUNSUPPORTED


def test_standalone_swiglu_kernel():
    """hs_swiglu (the unfused activation over a stored [T, 2F] gate | up tensor) against silu(g) * u in fp32
    from the same bf16 inputs, each element within its bf16 rounding."""
    from hybrid_serving_gb300._lib import check, lib
    g = torch.Generator(device="cuda").manual_seed(13)
    T, F = 333, 512
    gu = (torch.randn(T, 2 * F, device="cuda", generator=g) * 3).to(torch.bfloat16)
    out = torch.full((T, F), float("nan"), device="cuda", dtype=torch.bfloat16)
    check(lib.hs_swiglu(gu.data_ptr(), gu.stride(0), T, F, out.data_ptr(), out.stride(0),
                        torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    gt, up = gu[:, :F].float(), gu[:, F:].float()
    want = gt * torch.sigmoid(gt) * up
    err = (out.float() - want).abs()
    assert bool((err <= 2.0 ** -8 * want.abs() + 1e-6).all()), float(err.max())
