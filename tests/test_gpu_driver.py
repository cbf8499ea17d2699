"""Multi-segment driver on the GPU against the oracle: every attention call it
makes matches the oracle on the inputs it was given, the memory each call saw
is the oracle's Tail_M roll of the earlier segments (bit-exact), and a
checkpoint taken between segments resumes to identical results."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu

WL = W.WORKLOADS["seg128_bf16"].with_(B=2, H=2, L=128, M=128, layers=2, segments=3)


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy()


def make_driver(record, overlap=False):
    dev = torch.device("cuda")
    params = W.make_params(WL)
    mems = [m.to(dev, WL.torch_dtype) for m in W.initial_memories(WL)]
    rks = [W.project_r(lw, WL.M, WL.L, WL.H, device=dev) for lw in params.layers]
    drv = txl.SegmentDriver(mems, mem_stream=torch.cuda.Stream() if overlap else None)

    def project(n, mem, h):
        ci = W.call_inputs(WL, params.layers[n], params, mem, h, r_k32=rks[n])
        if record is not None:
            record.append({"n": n, "mem": mem.clone(), "h": h.clone(), "ci": ci})
        return ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale

    def next_input(n, out):
        if record is not None:
            record[-1]["out"] = out.clone()
        return W.merge_heads(out).to(WL.torch_dtype)

    return drv, project, next_input


@pytest.mark.parametrize("overlap", [False, True])
def test_driver_calls_and_memories_match_oracle(overlap):
    """overlap=True runs the rolls on a second stream."""
    rec = []
    drv, project, next_input = make_driver(rec, overlap)
    ref_mem = [bits(m) for m in drv.mems]
    for s in range(WL.segments):
        h0 = W.segment_input(WL, s).cuda().to(WL.torch_dtype)
        drv.run_segment(h0, project, next_input)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    assert len(rec) == WL.segments * WL.layers
    for c in rec:
        n = c["n"]
        # the memory this call attended to is the oracle's roll of the earlier segments
        assert np.array_equal(bits(c["mem"]), ref_mem[n])
        ref_mem[n] = oracle.mem_update(ref_mem[n], bits(c["h"]), WL.M)
        ci = c["ci"]
        cpu = [t.cpu() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
        ref = oracle.attn(*cpu, ci.scale)
        got = c["out"].float().cpu().double().numpy()
        tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
        assert np.abs(got - ref).max() <= tol
    for n, m in enumerate(drv.mems):
        assert np.array_equal(bits(m), ref_mem[n])


@pytest.mark.parametrize("overlap", [False, True])
def test_driver_checkpoint_resume_is_identical(overlap):
    drv, project, next_input = make_driver(None, overlap)
    h = [W.segment_input(WL, s).cuda().to(WL.torch_dtype) for s in range(3)]
    drv.run_segment(h[0], project, next_input)
    sd = drv.state_dict()
    a = drv.run_segment(h[1], project, next_input).clone()
    mem_a = [m.clone() for m in drv.mems]
    drv.load_state_dict(sd)
    assert drv.segments_done == 1
    b = drv.run_segment(h[1], project, next_input)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    for x, y in zip(mem_a, drv.mems):
        assert torch.equal(x, y)
