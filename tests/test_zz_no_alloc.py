"""The no-allocation key-split entry point (fa_fwd_split_noalloc) against the existing one and the oracle.

fa_fwd_split_noalloc serves callers that cannot allocate device memory when they call (a plug-in
whose host owns the GPU's memory, a serving loop that must not stall on an allocation): its
split partials live in a fixed scratch array inside the library instead of a caller workspace.
This file is collected last on purpose, so that a run stopping at the first failure has already
run everything else; it passes alone in a fresh process as well as after the other tests.
"""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_split_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_13_gb300 as ea
    from oracle import oracle
    from tests.parity import compare
    from workloads import random_inputs

    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    # calls in a row with different problems: the shared scratch keeps each call's partials, which
    # must not leak into the next call's result -- a smaller problem after a larger one, then a
    # larger one with more splits after a smaller one, so that stale partials sit where the new
    # call reads
    cases = [(6001, True, 3, 1, 2, 1000, 128), (6002, False, 2, 1, 2, 777, 64),
             (6003, True, 4, 2, 4, 2000, 128)]
    for seed, causal, splits, B, H, N, d in cases:
        inp = random_inputs(B, H, N, d, "bf16", seed=seed)
        q, k, v = (getattr(inp, n).to(dev) for n in "qkv")
        ref_o, ref_l = ea.fwd(q, k, v, causal=causal, num_splits=splits)  # caller workspace
        o = torch.empty_like(ref_o)
        lse = torch.empty_like(ref_l)
        rc = ea.fa_fwd_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, N, d, 1.0 / math.sqrt(d), causal,
                                     ea.FA_DTYPE_BF16, splits, stream=stream)
        assert rc == ea.FA_OK, rc
        torch.cuda.synchronize()
        # the same kernels on the same bytes with the same partials layout: bit-identical
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), (seed, splits)
        o_ref, l_ref = oracle.attention_fwd_inputs(inp, 1.0 / math.sqrt(d), causal)
        compare(o, lse, o_ref, l_ref, "bf16", f"no-alloc split {splits} (seed {seed})")
    assert ea.device_status(clear=True) == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_13_gb300 as ea

    B, H, N, d, splits = 1, 8, 32768, 128, 2
    assert ea.split_workspace_bytes(B, H, N, d, splits) > 64 << 20
    fake = 0x10000  # never dereferenced: the size check refuses the call before any launch
    rc = ea.fa_fwd_split_noalloc(fake, fake, fake, fake, fake, B, H, N, d, 0.1, 0,
                                 ea.FA_DTYPE_BF16, splits)
    assert rc == ea.FA_ERR_UNSUPPORTED
