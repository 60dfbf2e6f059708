"""The library inside a CUDA graph. The entry points enqueue work on the
caller's stream and never allocate or synchronise, so one forward + backward
can be captured and replayed; replays with new input values (copied into the
captured buffers) give the eager results bit for bit (dQ of the one-pass
backward, summed with fp32 atomics, to one bf16 ulp). The split forward is
captured too (its workspace allocated before the capture)."""
import pytest
import torch

from parity import assert_same_up_to_atomics

from exact_io_aware_attention_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def fa():
    import exact_io_aware_attention_gb300 as m
    return m


@pytest.mark.parametrize("d,algo", [(128, "fused"), (128, "split"), (256, "split")])
def test_forward_backward_graph_replays_match_eager(d, algo):
    B, H, N = 2, 4, 1000
    first = gen.make_inputs(B, H, N, d, case=990)
    q, k, v, do = (first[t].cuda() for t in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa().backward_workspace_bytes(B, H, N, d, algo), dtype=torch.uint8,
                     device="cuda")

    def step():
        fa().forward(q, k, v, causal=True, out=o, lse=lse)
        fa().backward(q, k, v, o, do, lse, causal=True, workspace=ws, dq=dq, dk=dk, dv=dv)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first calls (per-process kernel set-up) outside the capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for case in (991, 992):
        inp = gen.make_inputs(B, H, N, d, case=case)
        for t, dst in (("q", q), ("k", k), ("v", v), ("do", do)):
            dst.copy_(inp[t])
        graph.replay()
        torch.cuda.synchronize()
        got = [x.clone() for x in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        assert fa().device_status() == 0
        for a, b in zip(got[:2] + got[3:], (o, lse, dk, dv)):
            assert torch.equal(a, b)
        if algo == "split":
            assert torch.equal(got[2], dq)
        else:  # dQ summed with fp32 atomics: the same up to one bf16 ulp
            assert_same_up_to_atomics(got[2], dq, "graph replay dq")


def test_split_forward_in_a_graph():
    B, H, Nq, Nk, d = 1, 8, 1, 8192, 128
    inp = gen.make_inputs(B, H, Nq, d, case=993, with_do=False, Nk=Nk)
    q, k, v = (inp[t].cuda() for t in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Nq, device="cuda")
    o_eager, lse_eager = fa().forward(q, k, v, causal=True, num_splits=6)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa().forward(q, k, v, causal=True, out=o, lse=lse, num_splits=6)
    graph.replay()
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    assert torch.equal(o, o_eager) and torch.equal(lse, lse_eager)


def test_exp2_rate_measurement_is_plausible():
    """The SFU rate probe behind the exponential-rate ceiling: ex2.approx
    operations per second, which per SM and clock (at most the maximum SM
    clock) lies between one per sub-partition and the FMA rate."""
    rate = fa().measure_exp2_rate()
    props = torch.cuda.get_device_properties(0)
    per_sm_per_ghz = rate / props.multi_processor_count / 1e9
    assert 4.0 * 0.5 <= per_sm_per_ghz <= 128.0 * 2.1, per_sm_per_ghz
