"""moe_permute_static: the permutation with the library's own fixed device
scratch, for callers that cannot pass a workspace (no allocator of their own,
or a loop that must not call cudaMalloc). Called through the C-ABI twice in a
row, its results must equal moe_permute's (a workspace the test allocates).
Collected last so a failure here comes after every other test has run."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(T, k, E):
    A = T * k
    return (torch.full((E,), -5, dtype=torch.int32, device=DEV), torch.full((E + 1,), -5, dtype=torch.int32, device=DEV),
            torch.full((A,), -5, dtype=torch.int32, device=DEV), torch.full((A,), -5, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV))


def _ids(T, k, E, seed):
    g = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)).to(DEV)


@pytest.mark.parametrize("T,k,E", [(64, 2, 8), (4096, 8, 256), (16384, 8, 256), (3000, 5, 1000)])
def test_static_scratch_matches_workspace_version(cuda_lib, T, k, E):
    pqe = cuda_lib
    for call, seed in enumerate((T + E, T + E + 1)):   # two calls in a row, different inputs
        ids = _ids(T, k, E, seed)
        ref = _outputs(T, k, E)
        ws = torch.zeros(pqe.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
        pqe.moe_permute(ids, T, k, E, *ref[:4], ws, ref[4])
        got = _outputs(T, k, E)
        pqe.moe_permute_static(ids, T, k, E, *got)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b), (call, T, k, E)


def test_static_scratch_on_a_trace_and_capacity(cuda_lib):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["decode"]
    import oracle
    logits = synth.routing_logits(cfg, 64, 1)
    ids_np, _ = oracle.topk_gates(logits, cfg.k)
    ids = torch.from_numpy(ids_np).to(DEV)
    for _ in range(2):
        got = _outputs(64, cfg.k, cfg.E)
        pqe.moe_permute_static(ids, 64, cfg.k, cfg.E, *got)
        torch.cuda.synchronize()
        ref = oracle.permute(ids_np, cfg.E)
        for a, b in zip(got[:4], ref):
            assert np.array_equal(a.cpu().numpy(), b)
    # beyond the fixed scratch: refused on the host, nothing launched
    words = pqe.lib().moe_permute_static_max_words()
    T_big = (words // 1000 + 1) * 2048
    with pytest.raises(pqe.PqeError) as ei:
        pqe.moe_permute_static(None, T_big, 1, 1000, *_outputs(1, 1, 1000)[:2], None, None, _outputs(1, 1, 1)[4])
    assert ei.value.code == pqe.PQE_ERR_CAPACITY
