"""The module-batch sizer (pqe_module_batch_size): the smallest accumulated
batch at which a layer's expert FFN stops being weight-bound, on the roofline
of given HBM and FP8 ceilings. Host-only, so these run without a GPU.

Pins: the returned T is the roofline knee itself (compute time reaches the
memory time at T, not one granule before), with the FLOP and byte counts
taken from the layer's definition (6 H I FLOP per row; the FP8 page once per
expert; per row the token's bf16 x shared by its k rows and its bf16
out_perm row); the knee moves the way the ceilings say it must.
"""
import pytest

import paged_quantized_expert_gb300 as pqe


def _times(T, E, k, H, I, bw_gbs, p_tflops):
    """Roofline times (s) of one layer step with T tokens spread evenly over E experts."""
    rows = T * k
    flop = 6.0 * rows * H * I
    page = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    byts = E * page + T * H * 2 + rows * H * 2
    return flop / (p_tflops * 1e12), byts / (bw_gbs * 1e9)


@pytest.fixture(scope="module")
def lib():
    pqe.load()
    return pqe


@pytest.mark.parametrize("E,k,H,I", [(256, 8, 2048, 512), (512, 8, 2560, 640), (8, 2, 1024, 512), (64, 4, 1024, 256)])
@pytest.mark.parametrize("bw,p", [(6779.0, 3774.6), (8000.0, 4500.0), (3350.0, 1979.0)])
def test_knee_is_the_roofline_crossing(lib, E, k, H, I, bw, p):
    g = 1
    T = lib.pqe_module_batch_size(E, k, H, I, bw, p, g)
    assert T > 0
    c, m = _times(T, E, k, H, I, bw, p)
    assert c >= m * (1 - 1e-9)               # compute-bound at T
    c1, m1 = _times(T - g, E, k, H, I, bw, p)
    assert c1 < m1                            # still weight-bound one token earlier


def test_granule_rounds_up(lib):
    t1 = lib.pqe_module_batch_size(256, 8, 2048, 512, 6779.0, 3774.6, 1)
    t64 = lib.pqe_module_batch_size(256, 8, 2048, 512, 6779.0, 3774.6, 64)
    assert t64 % 64 == 0 and t1 <= t64 < t1 + 64


def test_knee_moves_with_the_ceilings(lib):
    base = lib.pqe_module_batch_size(256, 8, 2048, 512, 6779.0, 3774.6, 1)
    # more tensor throughput needs more rows per expert to keep it busy
    assert lib.pqe_module_batch_size(256, 8, 2048, 512, 6779.0, 4500.0, 1) > base
    # more bandwidth makes the weights cheaper: the knee comes earlier
    assert lib.pqe_module_batch_size(256, 8, 2048, 512, 8000.0, 3774.6, 1) < base
    # twice the experts over the same routing need twice the tokens
    e2 = lib.pqe_module_batch_size(512, 8, 2048, 512, 6779.0, 3774.6, 1)
    assert abs(e2 - 2 * base) <= 2


def test_invalid_arguments_and_no_knee(lib):
    f = lib.pqe_module_batch_size
    assert f(0, 8, 2048, 512, 6779.0, 3774.6, 64) == 0
    assert f(256, 0, 2048, 512, 6779.0, 3774.6, 64) == 0
    assert f(4, 8, 2048, 512, 6779.0, 3774.6, 64) == 0     # k > E
    assert f(256, 8, 100, 512, 6779.0, 3774.6, 64) == 0    # H not a multiple of 64
    assert f(256, 8, 2048, 512, 0.0, 3774.6, 64) == 0
    assert f(256, 8, 2048, 512, 6779.0, -1.0, 64) == 0
    assert f(256, 8, 2048, 512, 6779.0, 3774.6, 0) == 0
    # activations alone slower than the tensor cores (tiny I, huge peak): no knee
    assert f(256, 8, 2048, 64, 6779.0, 100000.0, 64) == 0
