"""The stream contract of the C ABI: every call enqueues its work on the
stream it is given and on no other. The current (default) stream is held busy
by a bounded sleep kernel while calls are issued on a non-blocking side
stream; they must finish before the sleep does, and give the same result as
on the default stream."""

import time

import pytest
import torch

from tpmlp_inputs import AttnWorkload, Workload, make_attn_inputs, make_block_inputs, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import tensor_transformer_mlp_column_gb300 as tp

    torch.cuda.set_device(0)
    return tp


def _finishes_while_default_stream_sleeps(fn):
    side = torch.cuda.Stream()  # PyTorch's pool streams do not synchronise with the default stream
    torch.cuda.synchronize()
    torch.cuda._sleep(4_000_000_000)  # about two seconds on the default stream (a bounded spin)
    done = torch.cuda.Event()
    with torch.cuda.stream(side):
        out = fn(side)
        done.record(side)
    t0 = time.time()
    while not done.query() and time.time() - t0 < 1.0:
        time.sleep(0.001)
    finished = done.query()
    torch.cuda.synchronize()
    return finished, out


def test_calls_run_on_the_given_stream(tp):
    w = Workload("s", 512, 256, 1024, 4, "bf16", 1.0, 0.05, 0.05, 1.0, True)
    d = {k: v.cuda() for k, v in make_inputs(w, seed=81).items()}
    sh = tp.tpmlp_shard(d["A"], d["B"], w.N)
    bi = {k: v.cuda() for k, v in make_block_inputs(w, seed=82).items()}
    shb = tp.tpmlp_shard(bi["A"], bi["B"], w.N)
    aw = AttnWorkload("sa", 2, 256, 256, 4, 2, "bf16", 1.0, 0.06)
    ai = {k: v.cuda() for k, v in make_attn_inputs(aw, seed=83).items()}
    sha = tp.tpmlp_attn_shard(ai["Wq"], ai["Wk"], ai["Wv"], ai["Wo"], aw.heads, aw.N)
    calls = {
        "forward faithful": lambda s: tp.tpmlp_forward(d["X"], sh, "faithful", stream=s),
        "forward fused": lambda s: tp.tpmlp_forward(d["X"], sh, "fused", stream=s),
        "backward": lambda s: tp.tpmlp_backward(d["X"], d["dY"], sh, "faithful", stream=s)[0],
        "block forward": lambda s: tp.tpmlp_block_forward(bi["x"], shb, "fused", stream=s),
        "attention": lambda s: tp.tpmlp_attn_forward(ai["X"], aw.batch, sha, "faithful", stream=s),
    }
    for name, fn in calls.items():
        ref = fn(torch.cuda.current_stream())
        torch.cuda.synchronize()
        finished, out = _finishes_while_default_stream_sleeps(fn)
        assert finished, f"{name}: waited for the default stream"
        assert torch.equal(out, ref), f"{name}: differs on the side stream"
    tp.tpmlp_check_status()


def test_concurrent_host_threads(tp):
    """Calls from several host threads, each with its own stream, workspace and
    shards, interleave freely: every thread's results equal the ones computed
    alone (the library's host state is per thread or set once per process)."""
    import threading

    shapes = [(2048, 1024, 4096, 4), (1000, 512, 2048, 8), (300, 256, 1024, 2)]
    jobs = []
    for i, (T, D, F, N) in enumerate(shapes):
        inp = {k: v.cuda() for k, v in make_inputs(Workload(f"thr{i}", T, D, F, N, "bf16", 1.0, 0.03, 0.03),
                                                    seed=90 + i).items()}
        sh = tp.tpmlp_shard(inp["A"], inp["B"], N)
        ref = {m: tp.tpmlp_forward(inp["X"], sh, m).clone() for m in ("faithful", "fused")}
        jobs.append((inp, sh, ref))
    torch.cuda.synchronize()
    errors = []

    def run(job):
        inp, sh, ref = job
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(20):
                    for m in ("faithful", "fused"):
                        Y = tp.tpmlp_forward(inp["X"], sh, m, stream=s)
                        s.synchronize()
                        if not torch.equal(Y, ref[m]):
                            errors.append(f"{m} differs in a concurrent thread")
                            return
        except Exception as e:  # reported below, on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert not any(t.is_alive() for t in threads)
    tp.tpmlp_check_status()
