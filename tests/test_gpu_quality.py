"""GPU parity of the 4-bit quality proxy (pqe_expert_quant_error): one expert's
FP8 and MXFP4 pages run on sampled tokens through the layer's own FFN kernels;
the sums (sum ||y4 - y8||^2, sum ||y8||^2) are compared with the oracle's fp64
values. 8 tokens take the weight stream (exact bf16 activations), 16 or 32
the tensor-core path (activations rounded per row to E4M3 for both pages, so
the two outputs' rounding errors are largely shared)."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("H,I,n,tol", [(256, 128, 8, 0.005), (256, 128, 32, 0.03), (2048, 512, 16, 0.03)])
def test_quant_error_matches_oracle(cuda_lib, orc, H, I, n, tol):
    pqe = cuda_lib
    cfg = synth.small_config(E=1, H=H, I=I, k=1, T=n, cid=93)
    w13, w2 = synth.expert_weights(cfg, 0)
    p8 = torch.zeros(pqe.slot_stride(H, I), dtype=torch.uint8, device=DEV)
    pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(DEV), torch.from_numpy(w2).to(DEV), H, I, p8)
    p4 = torch.zeros(pqe.page_bytes(pqe.PQE_FMT_MXFP4, H, I), dtype=torch.uint8, device=DEV)
    pqe.pqe_pack_mxfp4_page(p8, H, I, p4)
    x = synth.activations(cfg, n)
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    ws = torch.zeros(pqe.pqe_quality_workspace_size(n, H, I), dtype=torch.uint8, device=DEV)
    sums = torch.zeros(2, dtype=torch.float64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pqe.pqe_expert_quant_error(xd, n, p8, p4, H, I, sums, ws, status)
    torch.cuda.synchronize()
    first = sums.cpu().numpy().copy()
    assert status.item() == 0
    # a second call on the same workspace: the same sums (deterministic order)
    pqe.pqe_expert_quant_error(xd, n, p8, p4, H, I, sums, ws, status)
    torch.cuda.synchronize()
    assert np.array_equal(sums.cpu().numpy(), first)

    q13, s13 = orc.quant_e4m3_rows(w13)
    q2, s2 = orc.quant_e4m3_rows(w2)
    w8 = (q13, s13, q2, s2)
    w4 = orc.quant_mxfp4_rows(q13, s13) + orc.quant_mxfp4_rows(q2, s2)
    d2, r2 = orc.quant_error_sums(x, w8, w4, I)
    assert first[1] == pytest.approx(r2, rel=2e-2)
    err_gpu, err_ref = np.sqrt(first[0] / first[1]), np.sqrt(d2 / r2)
    assert 0 < err_ref < 1 and abs(err_gpu - err_ref) <= tol, (err_gpu, err_ref)


def test_quant_error_rejects_bad_arguments(cuda_lib):
    pqe = cuda_lib
    H, I, n = 256, 128, 4
    ws = torch.zeros(pqe.pqe_quality_workspace_size(n, H, I), dtype=torch.uint8, device=DEV)
    sums = torch.zeros(2, dtype=torch.float64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x = torch.zeros((n, H), dtype=torch.bfloat16, device=DEV)
    p8 = torch.zeros(pqe.slot_stride(H, I), dtype=torch.uint8, device=DEV)
    small = ws[: ws.numel() // 2]
    with pytest.raises(RuntimeError):
        pqe.pqe_expert_quant_error(x, n, p8, p8, H, I, sums, small, status)
    with pytest.raises(RuntimeError):
        pqe.pqe_expert_quant_error(x, n, p8, p8, 100, I, sums, ws, status)
