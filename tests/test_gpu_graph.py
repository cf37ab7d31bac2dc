"""Every library call is asynchronous on the caller's stream and can be
captured in a CUDA graph (the serving engines the pages describe replay whole
steps as graphs).

For each format pair: quantize W once, then capture quantize-X + GEMM (or the
GEMM alone when X stays bf16) into a graph on preallocated buffers.  Replaying
the graph after new X values are copied into the same input buffer must give,
bit for bit, what the eager calls give on those values (the kernels are
deterministic), and differ from the first input's result.  The same calls on a
side stream, ordered only by events, give the same bits again, and so do
several host threads driving the library at once on their own streams, in a
warm process and in a fresh one whose first calls all come from those threads.
"""
import pytest
import torch

from serving_amax_reduce_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = [
    # name, weight format, activation format, scale layout, M, N, K
    ("fp8_tensor", "FP8_TENSOR", "FP8_TENSOR", "CANONICAL", 200, 512, 384),
    ("fp8_block_token", "FP8_BLOCK128", "FP8_TOKEN", "CANONICAL", 256, 640, 512),
    ("fp8_block_group128", "FP8_BLOCK128", "FP8_GROUP128", "CANONICAL", 130, 384, 256),
    ("mxfp8", "MXFP8", "MXFP8", "MMA", 300, 512, 512),
    ("mxfp4", "MXFP4", "MXFP4", "MMA", 130, 384, 512),
    ("mxfp4_dual", "MXFP4_DUAL", "MXFP4_DUAL", "MMA", 130, 384, 1024),
    ("nvfp4", "NVFP4", "NVFP4", "MMA", 300, 640, 512),
    ("int8", "INT8_ROW", "INT8_ROW", "CANONICAL", 130, 640, 272),
    ("fp8_tensor_fused_x", "FP8_TENSOR", "BF16", "CANONICAL", 77, 640, 1040),
    ("w4a16_warp_mma", "INT4_G128_ASYM", "BF16", "CANONICAL", 1, 4096, 4096),
    ("w4a16_tcgen05", "INT4_G128_SYM", "BF16", "CANONICAL", 64, 256, 1024),
]


@pytest.fixture(scope="module")
def q():
    from gpu_util import require_gpu
    return require_gpu()


class Layer:
    """One quantized linear on preallocated buffers: run() enqueues
    quantize-X (if X is quantized) and the GEMM on the current stream."""

    def __init__(self, q, wname, xname, lname, M, N, K):
        self.q, self.M, self.N, self.K = q, M, N, K
        self.wf, self.xf, self.lay = q.Fmt[wname], q.Fmt[xname], q.Layout[lname]
        w = inputs.normal_bf16((N, K), 0.02, 201).to(DEV)
        self.bw = q.quantize_weight(self.wf, w, self.lay)
        self.xin = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
        self.bias = inputs.normal_bf16((1, N), 0.05, 202)[0].to(DEV)
        self.bx = None if self.xf == q.Fmt.BF16 else q.alloc_quant(self.xf, M, K, self.lay, DEV)
        self.y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

    def run(self):
        q = self.q
        kw = {"layout": self.lay, "bias": self.bias, "y": self.y, "w_global": self.bw.get("global"),
              "w_zeros": self.bw.get("zeros")}
        if self.bx is None:
            xa, xs = self.xin, None
        else:
            q.quantize_act(self.xf, self.xin, self.lay, bufs=self.bx)
            xa, xs = self.bx["codes"], self.bx["scales"]
            kw["x_global"] = self.bx.get("global")
        q.gemm(self.wf, self.xf, self.M, self.N, self.K, xa, xs, self.bw["codes"], self.bw["scales"], **kw)


@pytest.mark.parametrize("name,wname,xname,lname,M,N,K", CASES, ids=[c[0] for c in CASES])
def test_graph_replay_and_side_stream_match_eager(q, name, wname, xname, lname, M, N, K):
    layer = Layer(q, wname, xname, lname, M, N, K)
    x1 = inputs.normal_bf16((M, K), 1.0, 203).to(DEV)
    x2 = inputs.normal_bf16((M, K), 3.0, 204).to(DEV)

    # eager, default stream
    layer.xin.copy_(x1)
    layer.run()
    torch.cuda.synchronize()
    y1 = layer.y.clone()
    layer.xin.copy_(x2)
    layer.run()
    torch.cuda.synchronize()
    y2 = layer.y.clone()
    assert not torch.equal(y1.view(torch.int16), y2.view(torch.int16))

    # captured once, replayed on new contents of the same input buffer
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.run()
    for xv, yv in ((x1, y1), (x2, y2), (x1, y1)):
        layer.xin.copy_(xv)
        layer.y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(layer.y.view(torch.int16), yv.view(torch.int16)), "graph replay differs from eager"

    # a side stream, ordered against the default stream by events only
    side = torch.cuda.Stream()
    layer.xin.copy_(x2)
    layer.y.zero_()
    ready = torch.cuda.Event()
    ready.record()
    with torch.cuda.stream(side):
        side.wait_event(ready)
        layer.run()
        done = torch.cuda.Event()
        done.record(side)
    torch.cuda.current_stream().wait_event(done)
    torch.cuda.synchronize()
    assert torch.equal(layer.y.view(torch.int16), y2.view(torch.int16)), "side-stream result differs"
    assert q.read_device_status() == 0



def _threads_run(layers, reps):
    """Every layer on its own host thread and stream, all released at once;
    returns the exceptions the threads raised."""
    import threading

    start, errors = threading.Barrier(len(layers)), []

    def work(layer):
        try:
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(reps):
                    layer.y.zero_()
                    layer.run()
            s.synchronize()
        except Exception as e:       # reported by the caller, from the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(lay,)) for lay in layers]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    return errors


# FP8 block x per-token twice (two threads on one kernel), NVFP4, W4A16 on tcgen05
THREAD_CASES = [CASES[1], CASES[1], CASES[6], CASES[10]]


def _thread_layers(q):
    layers = []
    for j, (_, wname, xname, lname, M, N, K) in enumerate(THREAD_CASES):
        layer = Layer(q, wname, xname, lname, M, N, K)
        layer.xin.copy_(inputs.normal_bf16((M, K), 1.0, 205 + j).to(DEV))
        layers.append(layer)
    return layers


def test_host_threads_on_own_streams(q):
    """Several host threads drive the library at once (ctypes releases the GIL
    around each call), each on its own stream and buffers; every result equals
    the one computed alone."""
    layers = _thread_layers(q)
    want = []
    for layer in layers:
        layer.run()
        torch.cuda.synchronize()
        want.append(layer.y.clone())
    errors = _threads_run(layers, 20)
    assert not errors, errors
    for layer, y in zip(layers, want):
        assert torch.equal(layer.y.view(torch.int16), y.view(torch.int16))
    assert q.read_device_status() == 0


_COLD_CHILD = """
import sys, torch
sys.path[:0] = [sys.argv[1], sys.argv[2]]
import test_gpu_graph as T
from gpu_util import require_gpu
q = require_gpu()
layers = T._thread_layers(q)
errors = T._threads_run(layers, 3)          # the first call of every kernel happens here, on four threads
assert not errors, errors
got = [lay.y.clone() for lay in layers]
for lay, y in zip(layers, got):
    lay.y.zero_()
    lay.run()
    torch.cuda.synchronize()
    assert torch.equal(lay.y.view(torch.int16), y.view(torch.int16)), "threaded first calls differ"
assert q.read_device_status() == 0
print("ok")
"""


def test_first_calls_from_several_threads(q):
    """The library's one-time setups (device queries, the tensor-map encoder
    lookup, kernel attributes) run on whichever thread calls first: in a fresh
    process whose first calls all come from four threads at once, the results
    equal the serial ones."""
    import os
    import subprocess
    import sys

    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _COLD_CHILD, here, os.path.dirname(here)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
