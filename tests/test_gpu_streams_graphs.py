"""Forward and backward enqueued on a side stream, and captured in a CUDA graph and replayed.

Every entry point enqueues on the stream it is given and allocates nothing, so it can run on
any stream and inside stream capture. The shapes reach every kind of launch the forward and
backward make: no split; the forward's key ranges in a 4-CTA cluster with the dQ pass split
into 5 key ranges (float32 partial sums and a combine kernel); the dK/dV pass's query ranges
in a 4-CTA cluster; the one-pass backward at head size 64. The outputs equal those of the
same calls made eagerly on the default stream, bit for bit, except the one-pass kernel's dQ,
whose float32 additions land in any order (`check_reordered_sum`).
"""
import math

import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from tests import gpu_util as G
from tests.split_rules import dkv_query_splits, dq_key_splits, fwd_key_splits, one_pass
from tests.tolerance import check_reordered_sum

pytestmark = pytest.mark.gpu

# name: (bh, n_q, n_k, d)
SHAPES = {
    "plain": (4, 600, 700, 128),
    "fwd_and_dq_split": (1, 300, 5000, 64),
    "dkv_split": (2, 4096, 128, 128),
    "one_pass": (80, 256, 384, 64),
}


def test_the_shapes_reach_every_launch_kind():
    plain, fd, dkv, op = (SHAPES[n] for n in ("plain", "fwd_and_dq_split", "dkv_split", "one_pass"))
    assert fwd_key_splits(*plain) == 1 and dkv_query_splits(*plain) == 1 and dq_key_splits(*plain[:3]) == 1
    assert fwd_key_splits(*fd) == 4 and dq_key_splits(*fd[:3]) == 5 and not one_pass(fd[0], fd[2], fd[3])
    assert dkv_query_splits(*dkv) == 4
    assert one_pass(op[0], op[2], op[3])


class _Problem:
    """Inputs, outputs and workspace of one forward + backward, allocated once."""

    def __init__(self, name):
        torch = G.require_gpu()
        self.name = name
        bh, n_q, n_k, d = SHAPES[name]
        q, k, v = G.inputs(f"streams/{name}", bh, n_q, n_k, d, "bf16")
        d_o = synth.tensor(f"streams/{name}/do", (bh, n_q, d), "bf16")
        self.ins = [G.to_device(x, "bf16") for x in (q, k, v, d_o)]
        self.o = G.empty((bh, n_q, d), "bf16")
        self.lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
        self.grads = [G.empty(tuple(x.shape), "bf16") for x in self.ins[:3]]
        nbytes = binding.fa2_backward_workspace_size(bh, n_q, n_k, d, binding.DTYPE_BF16)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.scale = 1 / math.sqrt(d)

    def run(self, stream=None):
        qd, kd, vd, dod = self.ins
        binding.fa2_forward(qd, kd, vd, self.o, self.lse, self.scale, stream=stream)
        binding.fa2_backward(qd, kd, vd, self.o, dod, self.lse, *self.grads, self.ws, self.scale, stream=stream)

    def outputs(self):
        return [t.clone() for t in (self.o, self.lse, *self.grads)]

    def assert_equal(self, got, want, where):
        torch = G.require_gpu()
        names = ("O", "LSE", "dQ", "dK", "dV")
        for name, a, b in zip(names, got, want):
            if name == "dQ" and self.name == "one_pass":
                check_reordered_sum(G.to_f64(a), G.to_f64(b), f"{self.name}: {where} dQ")
            else:
                assert torch.equal(a, b), f"{self.name}: {where} {name} differs from the eager default-stream call"


@pytest.mark.parametrize("name", list(SHAPES))
def test_side_stream_equals_default_stream(name):
    torch = G.require_gpu()
    p = _Problem(name)
    p.run()
    torch.cuda.synchronize()
    want = p.outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for t in (p.o, p.lse, *p.grads):
        t.fill_(float("nan"))
    side.wait_stream(torch.cuda.current_stream())
    p.run(stream=side)
    side.synchronize()
    binding.fa2_device_status()
    p.assert_equal(p.outputs(), want, "side stream:")


@pytest.mark.parametrize("name", list(SHAPES))
def test_graph_capture_replays_the_calls(name):
    torch = G.require_gpu()
    p = _Problem(name)
    p.run()  # eager first: the library's one-time attribute settings happen outside capture
    torch.cuda.synchronize()
    want = p.outputs()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        p.run()  # enqueued on the capture stream (the binding takes torch's current stream)
    for _ in range(2):
        for t in (p.o, p.lse, *p.grads):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        binding.fa2_device_status()
        p.assert_equal(p.outputs(), want, "graph replay:")
