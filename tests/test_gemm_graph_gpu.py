"""CUDA graph capture of the C ABI's launches, against the oracle.

A graph replays the kernels, tensor maps and parameters it captured, reading
whatever the captured buffers hold at replay time.  Captured here, in one
graph on one stream: a one-CTA launch with one tile per CTA (eight epilogue
warps), one with several tiles per CTA (a batch), split-K over 2-CTA
clusters, wide CTA-pair tiles, 256 x 256 CTA-pair tiles with stream-K
(workspace grown on the stream before the capture; its counter reset is a
captured memset), and the allocation-free entry point.  Each replay follows
new operand values written into the same buffers and is compared with the
oracle element by element; integer inputs bit-exact.  A capture on a stream
without a stream-K workspace runs whole tiles (nothing is allocated during a
capture) and is just as exact.
"""
import numpy as np
import pytest
import torch

import shared_memory_operand_gb300 as smo
from synthetic import K_MAJOR, MN_MAJOR, make_problem
from tests.gemm_check import check, oracle_full

pytestmark = pytest.mark.gpu

_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    yield


# name -> (problem for a seed, planner knobs for this call, exact, entry point)
CASES = {
    "one_cta_one_tile": (lambda s: make_problem(1500, 1152, 896, a_major=K_MAJOR, b_major=MN_MAJOR,
                                                in_dtype="f16", out_dtype="f32", dist="uniform", seed=s),
                         {}, False, "ex"),
    "one_cta_batch": (lambda s: make_problem(300, 520, 200, batch=40, a_major=MN_MAJOR, b_major=K_MAJOR,
                                             out_dtype="bf16", dist="uniform", seed=s),
                      {"SMO_GEMM_FORCE_BN": "128"}, False, "ex"),
    "split_k": (lambda s: make_problem(512, 512, 4096, a_major=K_MAJOR, b_major=MN_MAJOR, out_dtype="f32",
                                       dist="int", seed=s),
                {}, True, "ex"),
    "wide_pair": (lambda s: make_problem(4096, 4096, 2048, a_major=K_MAJOR, b_major=MN_MAJOR,
                                         out_dtype="bf16", dist="uniform", seed=s),
                  {}, False, "ex"),
    "pair_stream_k": (lambda s: make_problem(2560, 2560, 1024, a_major=K_MAJOR, b_major=K_MAJOR,
                                             out_dtype="f32", dist="int", seed=s),
                      {"SMO_GEMM_FORCE_BN": "512", "SMO_GEMM_STREAM_K": "1"}, True, "ex"),
    "noalloc_pair": (lambda s: make_problem(2048, 2048, 256, a_major=K_MAJOR, b_major=MN_MAJOR,
                                            out_dtype="bf16", dist="uniform", seed=s),
                     {}, False, "noalloc"),
}


class _Dev:
    """Device buffers of one problem, reused by every replay."""

    def __init__(self, p):
        self.p = p
        self.A = p.A.cuda()
        self.B = p.B.cuda()
        self.C = torch.empty(p.c_numel(), dtype=_OUT[p.out_dtype], device="cuda")

    def launch(self, stream, entry):
        p = self.p
        fn = smo.gemm_ex_noalloc if entry == "noalloc" else smo.gemm_ex
        fn(self.A, p.lda, p.a_major, self.B, p.ldb, p.b_major, self.C, p.ldc, p.M, p.N, p.K,
           in_dtype=p.in_dtype, out_dtype=p.out_dtype, batch=p.batch, strideA=p.strideA,
           strideB=p.strideB, strideC=p.strideC, stream=stream)

    def reload(self, q):
        self.A.copy_(q.A)
        self.B.copy_(q.B)
        self.p = q

    def result(self):
        p = self.p
        c = self.C.cpu()
        stride = p.strideC if p.batch > 1 else p.M * p.ldc
        full = torch.as_strided(c, (p.batch, p.M, p.ldc), (stride, p.ldc, 1))
        return full[:, :, :p.N].to(torch.float64).numpy()


def _launch_all(devs, stream, monkeypatch):
    for name, d in devs.items():
        _, env, _, entry = CASES[name]
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        d.launch(stream, entry)
        for k in env:
            monkeypatch.delenv(k)


def _check_all(devs):
    for name, d in devs.items():
        check(d.p, d.result(), oracle_full(d.p), exact=CASES[name][2])


def _statuses(stream):
    return smo.gemm_check(stream), smo.gemm_check_noalloc(stream)


def test_graph_cases_reach_their_kernels(monkeypatch):
    n = torch.cuda.get_device_properties(0).multi_processor_count
    d = smo.gemm_plan_describe(1500, 1152, 896, K_MAJOR, MN_MAJOR, "f16", "f32", 1, n)
    assert not d["pair"] and not d["split"] and d["tiles"] <= d["grid"] and d["threads"] == 320
    d = smo.gemm_plan_describe(512, 512, 4096, K_MAJOR, MN_MAJOR, "bf16", "f32", 1, n)
    assert d["split"]
    d = smo.gemm_plan_describe(4096, 4096, 2048, K_MAJOR, MN_MAJOR, "bf16", "bf16", 1, n)
    assert d["wide"]
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "128")
    d = smo.gemm_plan_describe(300, 520, 200, MN_MAJOR, K_MAJOR, "bf16", "bf16", 40, n)
    assert not d["pair"] and d["tiles"] > d["grid"] and d["threads"] == 192
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "512")
    d = smo.gemm_plan_describe(2560, 2560, 1024, K_MAJOR, K_MAJOR, "bf16", "f32", 1, n)
    assert d["pair"] and not d["wide"] and d["tiles"] == 100      # a partial last wave: stream-K


def test_graph_capture_and_replay_with_new_inputs(monkeypatch):
    s = torch.cuda.Stream()
    devs = {name: _Dev(case[0](1)) for name, case in CASES.items()}
    # first launches outside the capture: kernel attributes, the stream-K
    # workspace of `s`, the allocation-free entry point's set-up
    _launch_all(devs, s, monkeypatch)
    assert _statuses(s) == (smo.GEMM_OK, smo.GEMM_OK)
    _check_all(devs)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _launch_all(devs, s, monkeypatch)
    for seed in (2, 3):
        for name, d in devs.items():
            d.reload(CASES[name][0](seed))
            d.C.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        assert _statuses(s) == (smo.GEMM_OK, smo.GEMM_OK)
        _check_all(devs)


def test_graph_capture_without_stream_k_workspace(monkeypatch):
    """A stream that never ran a stream-K launch has no workspace; during a
    capture none may be allocated, so the captured launch runs whole tiles."""
    s = torch.cuda.Stream()
    name = "pair_stream_k"
    d = _Dev(CASES[name][0](5))
    # the kernel's attributes are set by a launch on another stream, so that
    # only the workspace is missing on `s`
    warm = torch.cuda.Stream()
    _launch_all({name: d}, warm, monkeypatch)
    assert smo.gemm_check(warm) == smo.GEMM_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _launch_all({name: d}, s, monkeypatch)
    for seed in (6, 7):
        d.reload(CASES[name][0](seed))
        d.C.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        assert smo.gemm_check(s) == smo.GEMM_OK
        check(d.p, d.result(), oracle_full(d.p), exact=True)
    assert np.isfinite(d.result()).all()
