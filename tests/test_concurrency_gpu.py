"""Concurrent use of the library from several host threads.

Each thread has its own CUDA stream (torch's current stream is per thread)
and its own workspace; the library's shared host state (the tiling-plan
cache, the per-device information, the tensor-map encoder) is reached from
all of them at once.  Every kernel is deterministic, so each concurrent
result must equal, bit for bit, the same call made alone on the default
stream.  The calls mix forward scoring, K-candidate scoring, KL, the
backward and the block-scaled forward and KL on different shapes, so that
the threads also ask for different plans at the same time.
"""
import threading

import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads

pytestmark = pytest.mark.gpu
THREADS = 4
REPEATS = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _jobs():
    f = workloads.make(workloads.WORKLOADS[0].scaled(T=1000, H=1024, V=30000, seed=90), "cuda")
    p = workloads.make(workloads.WORKLOADS[2].scaled(T=3000, H=512, V=20000, seed=91), "cuda")
    k = workloads.make(workloads.WORKLOADS[3].scaled(T=700, H=768, V=25000, seed=92), "cuda")
    b = workloads.make(workloads.WORKLOADS[4].scaled(T=900, H=512, V=17000, seed=93), "cuda")
    cand = torch.stack([f["targets"], f["targets"].flip(0), (f["targets"] + 7) % 30000], 1)
    fhead = flp.mx_head_quantize(f["W"])
    khead = flp.mx_head_quantize(k["W_t"])
    return {
        "block-scaled forward": lambda: flp.logprob_entropy_mx(f["h"], fhead, 30000, f["targets"],
                                                               None, 0.8),
        "block-scaled kl": lambda: (flp.kl_divergence_mx(k["h_s"], k["W_s"], k["h_t"], khead),),
        "forward": lambda: flp.logprob_entropy(f["h"], f["W"], f["targets"], None, 0.8),
        "packed": lambda: flp.logprob_entropy(p["h"], p["W"], p["targets"], p["row_idx"], 1.0),
        "k-candidates": lambda: flp.logprob_entropy_k(f["h"], f["W"], cand, None, 0.8),
        "kl": lambda: (flp.kl_divergence(k["h_s"], k["W_s"], k["h_t"], k["W_t"]),),
        "backward": lambda: flp.backward(b["h"], b["W"], b["targets"], b["row_idx"], b["tau"],
                                         b["g1"], b["g2"]),
    }


def test_threads_with_own_streams_match_serial_results():
    jobs = _jobs()
    names = sorted(jobs)
    want = {}
    for name in names:
        want[name] = [t.clone() for t in jobs[name]()]
    torch.cuda.synchronize()

    errors = []
    start = threading.Barrier(THREADS)

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                for r in range(REPEATS):
                    name = names[(i + r) % len(names)]
                    got = jobs[name]()
                    stream.synchronize()
                    for a, b in zip(got, want[name]):
                        if not torch.equal(a, b):
                            errors.append("thread %d repeat %d: %s differs" % (i, r, name))
        except Exception as e:  # reported on the main thread
            errors.append("thread %d: %r" % (i, e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors


def test_calls_on_a_side_stream_are_ordered_after_its_producers():
    """Inputs written on a side stream and scored on that stream: the call is
    enqueued on the caller's current stream, so it sees the producer's writes
    without any synchronisation from the library."""
    f = workloads.make(workloads.WORKLOADS[0].scaled(T=600, H=512, V=9000, seed=94), "cuda")
    want = flp.logprob_entropy(f["h"], f["W"], f["targets"], None, 1.0)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        h = torch.empty_like(f["h"])
        torch.cuda._sleep(20_000_000)          # delay the copy: a race would read garbage
        h.copy_(f["h"])
        got = flp.logprob_entropy(h, f["W"], f["targets"], None, 1.0)
    side.synchronize()
    assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])
