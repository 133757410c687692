"""The no-allocation routing entry point (GPU).

Some callers cannot allocate device memory -- their framework's allocator
already owns the GPU, or they cannot accept the synchronisation an
allocation may cause.  moe_route_permute_static serves them: its scratch is
a fixed array inside the library.  This test calls it through the C ABI
twice in a row (different sizes, so stale scratch contents from the first
call would show) and checks each result against the regular entry point's
routing (moe_forward + moe_debug_routing) and against the oracle, at the
sizes the fixed array is built for (T = 4096, E = 512, K = 16) too: ids,
offsets and permutation bit-exact, routing weights within 1e-6.  It lives in
a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _regular_routing(s, T, logits):
    from moe_expert_layer_histogram_gb300 import MoELayer
    case = workloads.make_case(s, T=T, seed=4, device="cuda")
    layer = MoELayer(T, s["H"], s["I"], s["E"], s["K"], s["fmt"], s["clamp"])
    layer.prepare_weights(case["weights"])
    layer.forward(case["hidden"], logits)
    ids, w, off, perm = (t.cpu().numpy() for t in layer.routing())
    torch.cuda.synchronize()
    layer.close()
    return ids, w, off, perm


def _static_routing(T, E, K, logits):
    from moe_expert_layer_histogram_gb300 import moe_route_permute_static
    dev = torch.device("cuda")
    ids = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    w = torch.zeros(T, K, dtype=torch.float32, device=dev)
    off = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T * K,), -1, dtype=torch.int32, device=dev)
    moe_route_permute_static(logits, T, E, K, ids, w, off, perm,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), off.cpu().numpy(), perm.cpu().numpy()


def test_static_routing_matches_regular_entry_point_twice():
    s = workloads.spec("nvfp4_zipf_small", E=40, K=6)
    for T in (300, 70):                     # two calls in a row, second smaller
        logits = workloads.make_case(s, T=T, seed=T, device="cuda", weights=False)["logits"]
        ref = _regular_routing(s, T, logits)
        got = _static_routing(T, s["E"], s["K"], logits)
        assert np.array_equal(got[0], ref[0])
        assert np.max(np.abs(got[1] - ref[1])) <= 1e-6
        assert np.array_equal(got[2], ref[2])
        assert np.array_equal(got[3], ref[3])


def _check_vs_oracle(got, logits, K, E):
    lg = logits.cpu().numpy()
    ids_ref, w_ref = oracle.route(lg, K)
    off_ref, perm_ref, _ = oracle.permute(ids_ref, E)
    assert np.array_equal(got[0], ids_ref)
    assert np.max(np.abs(got[1] - w_ref)) <= 1e-6
    assert np.array_equal(got[2], off_ref)
    assert np.array_equal(got[3], perm_ref)


def test_static_routing_at_its_limits_matches_oracle_twice():
    # T = 4096 (64 routing blocks, the array's capacity), E = 512 (16 logits
    # per lane), K = 16; then a smaller call on the same array
    for T, E, K, seed in ((4096, 512, 16, 1), (70, 40, 6, 2), (4096, 512, 16, 3)):
        g = torch.Generator().manual_seed(seed)
        logits = torch.randn(T, E, generator=g).cuda()
        got = _static_routing(T, E, K, logits)
        _check_vs_oracle(got, logits, K, E)


def test_static_routing_rejects_sizes_beyond_its_scratch():
    from moe_expert_layer_histogram_gb300 import MoEError, moe_route_permute_static
    x = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(MoEError) as e:
        moe_route_permute_static(x, 4097, 8, 2, x, x, x, x)
    assert e.value.code == 2
    with pytest.raises(MoEError) as e:
        moe_route_permute_static(x, 16, 513, 2, x, x, x, x)
    assert e.value.code == 2
