"""Stream order under programmatic dependent launch.

Every kernel of the library may be scheduled while the previous kernel of
its stream finishes, and waits for that kernel before it touches global
memory.  These tests chain calls on one stream, each consuming (or
overwriting) what the previous one produced or read, with no host
synchronisation in between, and require results bit-identical to the same
calls made one at a time with strict ordering and a synchronisation after
each.  Every kernel family appears as both producer and consumer.
"""
import pytest
import torch

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build
from memory_bound_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STRICT = {"strict_order": 1}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def _input(M, N, dtype, seed, kind="normal1"):
    return W.generate(W.custom(M, N, dtype, seed=seed, kind=kind), "cuda")


def _with(opts, extra):
    o = dict(opts or {})
    o.update(extra)
    return o


PATHS = {
    "rows": {"path": rs.RS_PATH_ROWS},
    "ring": {"path": rs.RS_PATH_RING},
    "stream": {"path": rs.RS_PATH_STREAM},
    "cluster": {"path": rs.RS_PATH_CLUSTER},
}


def _chain(x, w, b, paths, strict):
    """softmax -> rmsnorm -> layernorm -> softmax, each on the previous output."""
    outs = []
    cur = x
    steps = [("sm", paths[0]), ("rms", paths[1]), ("ln", paths[2]), ("sm", paths[3])]
    for op, p in steps:
        opts = _with(PATHS[p], STRICT) if strict else dict(PATHS[p])
        if op == "sm":
            y = rs.softmax(cur, options=opts)
        elif op == "rms":
            y = rs.rmsnorm(cur, w, eps=1e-6, options=opts)
        else:
            y = rs.layernorm(cur, w, b, eps=1e-5, options=opts)
        if strict:
            torch.cuda.synchronize()
        outs.append(y)
        cur = y
    return outs


@pytest.mark.parametrize("paths", [("rows", "ring", "rows", "ring"), ("ring", "rows", "ring", "rows"),
                                   ("rows", "stream", "stream", "rows"), ("ring", "ring", "ring", "ring")])
def test_dependent_chain_matches_one_call_at_a_time(paths):
    M, N = 2048, 4096
    x = _input(M, N, "bf16", seed=7)
    w, b = W.norm_params(N, "bf16", 7, "cuda")
    for _ in range(3):
        fast = _chain(x, w, b, paths, strict=False)
        torch.cuda.synchronize()
        slow = _chain(x, w, b, paths, strict=True)
        for i, (f, s) in enumerate(zip(fast, slow)):
            assert torch.equal(f.view(torch.int16), s.view(torch.int16)), f"step {i} differs"


def test_cluster_kernels_in_a_dependent_chain():
    M, N = 64, 131072
    x = _input(M, N, "f16", seed=3, kind="normal_spike")
    a = rs.softmax(x, options={"path": rs.RS_PATH_CLUSTER})
    b = rs.softmax(a, options={"path": rs.RS_PATH_STREAM, "cluster_size": 4})
    c = rs.softmax(b, options={"path": rs.RS_PATH_CLUSTER, "ring_values": rs.RS_RING_REREAD})
    torch.cuda.synchronize()
    a2 = rs.softmax(x, options=_with({"path": rs.RS_PATH_CLUSTER}, STRICT))
    torch.cuda.synchronize()
    b2 = rs.softmax(a2, options=_with({"path": rs.RS_PATH_STREAM, "cluster_size": 4}, STRICT))
    torch.cuda.synchronize()
    c2 = rs.softmax(b2, options=_with({"path": rs.RS_PATH_CLUSTER, "ring_values": rs.RS_RING_REREAD}, STRICT))
    torch.cuda.synchronize()
    for f, s in [(a, a2), (b, b2), (c, c2)]:
        assert torch.equal(f.view(torch.int16), s.view(torch.int16))


@pytest.mark.parametrize("first,second", [("ring", "rows"), ("rows", "ring"), ("cluster", "rows"),
                                          ("rows", "cluster")])
def test_next_call_does_not_overwrite_what_the_previous_one_reads(first, second):
    # Call 1 reads x; call 2 writes its result into x.  Call 1's output must
    # be that of the original x.
    M, N = 512, 16384 if "cluster" in (first, second) else 4096
    x = _input(M, N, "bf16", seed=11)
    x0 = x.clone()
    z = _input(M, N, "bf16", seed=12)
    want = rs.softmax(x0, options=_with(PATHS[first], STRICT))
    torch.cuda.synchronize()
    for _ in range(3):
        x.copy_(x0)
        y = rs.softmax(x, options=PATHS[first])
        rs.softmax(z, out=x, options=PATHS[second])
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_host_copy_after_a_call_sees_the_result():
    x = _input(1024, 1024, "f32", seed=5)
    y = rs.softmax(x)
    host = y.cpu()  # a device-to-host copy right behind the kernel
    torch.cuda.synchronize()
    assert torch.equal(host, y.cpu())
