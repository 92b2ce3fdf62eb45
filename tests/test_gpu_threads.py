"""Library calls from several host threads at once (GPU).

Each thread has its own plan, buffers and CUDA stream; the plans walk several
chunks (a host read of the tile count per call) and fork side streams, so
those paths run concurrently.  The results equal a serial run's: losses bit
for bit (the forward has no atomics), gradients to 1e-5 (their reductions
are atomic, so the summation order may differ).  A profiling session open
meanwhile counts the launches of both threads.
"""
import threading

import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import synthetic
from tests.helpers import rel_l2, to_device

pytestmark = pytest.mark.gpu

REPS = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def _case(seed, dtype):
    inp = synthetic.custom(B=4, T=40, U=9, HA=64, HL=64, H=64, V=256, dtype=dtype, seed=seed,
                           bias_std=0.2)
    dev = to_device(inp)
    r = rn.Rnnt.for_inputs(inp, tile_cells=128 * 3)  # 3 tiles per chunk: several chunks
    assert rn.rnnt_graph_capturable(r.dims) == 0
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    return r, args


def _run(r, args, stream, out):
    with torch.cuda.stream(stream):
        for _ in range(REPS):
            loss = r.fwd(*args, stream=stream)
            g = r.bwd(*args, stream=stream)
            out.append((loss.clone(), {k: v.clone() for k, v in g.items()}))
    stream.synchronize()


def _launches(prof):
    return sum(n for _, n in prof.values())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_concurrent_calls_from_two_threads(dtype):
    cases = [_case(81, dtype), _case(82, dtype)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    # serial reference, profiled
    ref = [[], []]
    rn.rnnt_profile_start(1 << 16)
    for i in range(2):
        _run(*cases[i], streams[i], ref[i])
    serial_launches = _launches(rn.rnnt_profile_stop())

    # the same work from two threads at once, profiled
    got = [[], []]
    errors = []

    def worker(i):
        try:
            _run(*cases[i], streams[i], got[i])
        except Exception as e:  # reported by the main thread
            errors.append(e)

    rn.rnnt_profile_start(1 << 16)
    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    concurrent_launches = _launches(rn.rnnt_profile_stop())
    assert not errors, errors
    assert concurrent_launches == serial_launches

    for i in range(2):
        r = cases[i][0]
        assert r.status() == (0, 0)
        assert len(got[i]) == REPS
        for (l_ref, g_ref), (l_got, g_got) in zip(ref[i], got[i]):
            assert torch.equal(l_ref, l_got)
            for k in g_ref:
                assert rel_l2(g_got[k].double().cpu().numpy(),
                              g_ref[k].double().cpu().numpy()) < 1e-5, k
