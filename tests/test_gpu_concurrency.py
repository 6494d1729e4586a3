"""Serving-style use: calls from several host threads on their own streams at
once, and calls captured into a CUDA graph and replayed.  Results must be
those of the same calls made one at a time (bit for bit: same kernels, same
order)."""
import threading

import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def test_threads_on_their_own_streams():
    sizes = [(1 << 22) + 17 * k for k in range(8)]
    data = [synth.generate(n, "uniform_pm1", tcr.F16, seed=200 + k) for k, n in enumerate(sizes)]
    refs = [oracle.fixed_order(x, tcr.F16) for x in data]
    tensors = [torch.from_numpy(x.view(np.int16)).cuda() for x in data]
    torch.cuda.synchronize()
    errors = []

    def work(k):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = [tcr.tcr_reduce_sum(tensors[k], tcr.Mode(kind), stream=s)
                        for kind in (tcr.FIXED_ORDER, tcr.MMA_CHAIN, tcr.SHUFFLE_TREE)] * 1
                for _ in range(10):
                    o = tcr.tcr_reduce_sum(tensors[k], tcr.Mode(tcr.FIXED_ORDER), stream=s)
            s.synchronize()
            if o.cpu().numpy()[0].tobytes() != refs[k].tobytes():
                errors.append(f"thread {k}: {o.cpu().numpy()[0]!r} != {refs[k]!r}")
            if outs[0].cpu().numpy()[0].tobytes() != refs[k].tobytes():
                errors.append(f"thread {k}: first call differs")
        except Exception as e:        # reported below
            errors.append(f"thread {k}: {e!r}")

    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(sizes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_calls_captured_in_a_cuda_graph_replay_exactly():
    n = (1 << 24) + 5
    x = synth.generate(n, "normal", tcr.BF16, seed=210)
    t = torch.from_numpy(x.view(np.int16)).cuda()
    rows, cols = 4096, 3000
    xr = synth.generate(rows * cols, "normal", tcr.F16, seed=211).reshape(rows, cols)
    tr = torch.from_numpy(xr.reshape(-1).view(np.int16)).cuda().view(rows, cols)
    A = torch.from_numpy(synth.generate(512 * 1024, "normal", tcr.BF16, seed=212).view(np.int16))
    W = torch.from_numpy(synth.generate(640 * 1024, "normal", tcr.BF16, seed=213).view(np.int16))
    A = A.cuda().view(512, 1024).view(torch.bfloat16)
    W = W.cuda().view(640, 1024).view(torch.bfloat16)
    modes = [tcr.Mode(k, dtype=tcr.BF16) for k in (tcr.FIXED_ORDER, tcr.MMA_CHAIN, tcr.SHUFFLE_TREE,
                                                     tcr.MMA_CHAIN_TMEM)]
    sums = torch.zeros(len(modes), device="cuda")
    r_out = torch.zeros(rows, device="cuda")
    c_out = torch.zeros(512, 640, device="cuda")

    def step(stream):
        for i, m in enumerate(modes):
            tcr.tcr_reduce_sum(t, m, out=sums[i:i + 1], stream=stream)
        tcr.tcr_reduce_rows(tr, tcr.Mode(tcr.FIXED_ORDER), out=r_out, stream=stream)
        tcr.tcr_gemm_splitk(A, W, splits=4, out=c_out, stream=stream)

    # eager once (sets every per-device cache and kernel attribute), keep the bits
    step(None)
    torch.cuda.synchronize()
    eager = (sums.cpu().numpy().copy(), r_out.cpu().numpy().copy(), c_out.cpu().numpy().copy())
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sums.zero_()
        r_out.zero_()
        c_out.zero_()
        with torch.cuda.graph(g, stream=s):
            step(s)
    for _ in range(5):
        sums.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert sums.cpu().numpy().tobytes() == eager[0].tobytes()
    assert r_out.cpu().numpy().tobytes() == eager[1].tobytes()
    assert c_out.cpu().numpy().tobytes() == eager[2].tobytes()
    assert sums.cpu().numpy()[0] == oracle.fixed_order(x, tcr.BF16)
