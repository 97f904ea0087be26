"""Pipelined host steps give the results of plain sequential steps.

HostPipeline (fp8_paged_kv_gb300.pool) runs decode steps from pinned host
buffers with step i+1's inputs copied in and step i-1's results copied out
while step i runs, alternating two device I/O buffer pairs.  Each step's
results (out, lse, abort mask) must be the same bytes as the same step run
on its own through DecodePool.step, eagerly and when captured in a CUDA graph.
"""
import numpy as np
import pytest
import torch

from fp8_paged_kv_gb300.pool import DecodePool, HostPipeline
from workloads import custom

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("graph", [False, True])
def test_pipelined_steps_match_sequential_steps(fp8, graph):
    n = 6
    wl = custom(131, B=5, Hq=16, Hkv=2, ps=16, prompt_lens=[40, 0, 300, 17, 1000], steps=n)
    wl.expected_tags[2, 3] ^= np.uint32(1)          # request 2 fails the tag check
    pool = DecodePool(wl, fp8=fp8, device=DEV)
    pool.prefill()
    pool.count_aborts = False
    # reference: each step alone, its inputs uploaded, its results read back
    host_in, ref_out = [], []
    for s in range(n):
        pool.set_step(s)
        host_in.append(pool.io_in.cpu().pin_memory())
        pool.step(validate=True)
        torch.cuda.synchronize()
        ref_out.append(pool.io_out.cpu().clone())
    assert ref_out[0].numel() > 0
    host_out = [torch.full_like(r, 0xAB).pin_memory() for r in ref_out]
    pipe = HostPipeline(pool, host_in, host_out, validate=True)
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            pipe.run(n)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for h in host_out:
            h.fill_(0xAB)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pipe.run(n)
        g.replay()
    else:
        pipe.run(n)
    torch.cuda.synchronize()
    for s in range(n):
        assert torch.equal(host_out[s], ref_out[s]), f"step {s}"
    # the reference itself: request 2 aborted at every step, the others not
    off = pool._io[0][3]["abort_mask"].data_ptr() - pool._io[0][2].data_ptr()
    for s in range(n):
        assert ref_out[s][off:off + wl.B].tolist() == [0, 0, 1, 0, 0]
    assert pool.workspace[:4].view(torch.int32).item() == 0
