"""Shared-memory bank microbenchmark on the GPU against the oracle's bank
simulator: for access patterns the pages discuss (and the GEMM epilogue's own
stores), the measured cycles per access instruction must follow the number of
wavefronts the simulator predicts for the same per-lane offsets."""
import numpy as np
import pytest
import torch

import shared_memory_operand_gb300 as smo
from oracle import banksim
from tests.smem_patterns import PATTERNS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def measured():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    res = {}
    for name, (offs, nbytes) in PATTERNS.items():
        o = torch.tensor(offs, dtype=torch.int32, device="cuda")
        for store in (True, False):
            iters = 2048
            smo.smem_bank_probe(o, nbytes, store, iters, out)
            torch.cuda.synchronize()
            cyc = out[0].item() / (iters * 8)
            res[(name, store)] = (banksim.simulate(offs, nbytes).wavefronts, cyc)
    return res


def test_cycles_follow_predicted_wavefronts(measured):
    """cycles per access ~ a + b * predicted wavefronts over every pattern,
    loads and stores (linear fit R^2 >= 0.98; each point within 20 % or 2.5
    cycles of the fit), and never faster for more predicted wavefronts."""
    w = np.array([v[0] for v in measured.values()], dtype=float)
    c = np.array([v[1] for v in measured.values()], dtype=float)
    b, a = np.polyfit(w, c, 1)
    fit = a + b * w
    r2 = 1 - np.sum((c - fit) ** 2) / np.sum((c - c.mean()) ** 2)
    assert r2 >= 0.98, r2
    assert b > 0
    for (name, store), (wv, cyc) in measured.items():
        f = a + b * wv
        assert abs(cyc - f) <= max(0.2 * f, 2.5), (name, store, wv, cyc, f)
    order = np.argsort(w, kind="stable")
    for i, j in zip(order[:-1], order[1:]):
        if w[j] > w[i]:
            assert c[j] >= 0.9 * c[i]


def test_epilogue_swizzle_is_what_makes_the_stores_cheap(measured):
    sw = measured[("st16_epilogue_swizzled", True)]
    un = measured[("st16_epilogue_unswizzled", True)]
    lin = measured[("st16_linear", True)]
    assert sw[0] == 4 and un[0] == 32                    # simulator: 1-way vs 8-way
    assert abs(sw[1] / lin[1] - 1) < 0.1                 # as cheap as contiguous rows
    assert un[1] > 4.0 * sw[1]


def test_page_padding_ordering(measured):
    """[64][64+PAD] column reads on 32 banks: PAD 0 is the worst, PAD 32 next,
    PAD 1 / 2 / 4 all near the floor ("LDS Optimization", "Padding Amount")."""
    cyc = {p: measured[(f"ld2_pad{p}", False)][1] for p in (0, 1, 2, 4, 32)}
    assert cyc[0] > cyc[32] > 2 * max(cyc[1], cyc[2], cyc[4])


def test_tensor_peak_probe_runs_on_every_cluster():
    """Back-to-back tcgen05.mma.cta_group::2 on resident shared-memory tiles:
    every cluster finishes within its bounded wait, and the rate is that of a
    working tensor pipe (a loose floor; the value itself is reported by the
    bench)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    iters = 4000
    out = torch.full((2 * 1024,), -2, dtype=torch.int64, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    n = smo.tc_peak_probe(iters, out, 1024)
    e1.record()
    torch.cuda.synchronize()
    per = out[: 2 * n].view(n, 2).cpu()
    assert n >= 1 and torch.all(per[:, 0] > 0) and torch.all(per[:, 1] > 0)
    flops = n * iters * 4 * 2.0 * 256 * 256 * 16
    tflops = flops / (e0.elapsed_time(e1) / 1e3) / 1e12
    assert tflops > 300.0, tflops


def _l2_rate(buf, iters, stages=6):
    out = torch.full((2 * 1024,), -2, dtype=torch.int64, device="cuda")
    smo.l2_read_probe(buf, buf.numel(), 50, out, 1024, stages)  # warm (and bring an L2-sized buffer in)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    n = smo.l2_read_probe(buf, buf.numel(), iters, out, 1024, stages)
    e1.record()
    torch.cuda.synchronize()
    per = out[: 2 * n].view(n, 2).cpu()
    assert n >= 1 and torch.all(per[:, 0] > 0) and torch.all(per[:, 1] > 0), "a bounded wait ran out"
    return n * iters * 32768 / (e0.elapsed_time(e1) / 1e3)


def test_l2_read_probe_runs_and_l2_outpaces_hbm():
    """Bulk copies from global into shared memory on every SM, nothing else:
    every CTA finishes within its bounded waits; a 64 MiB buffer (resident in
    the 126 MB L2) streams faster than a 2 GiB one (from HBM), and the HBM rate
    is of the order of the measured copy bandwidth."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    small = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    big = torch.zeros(2 << 30, dtype=torch.uint8, device="cuda")
    l2 = _l2_rate(small, 2000)
    hbm = _l2_rate(big, 400)
    print(f"L2 -> SM {l2 / 1e12:.2f} TB/s, HBM -> SM {hbm / 1e12:.2f} TB/s")
    assert l2 > hbm > 2e12, (l2, hbm)
    # fewer copies in flight per SM, lower rate (Little's law: rate = bytes in flight / latency)
    by_stages = {s: _l2_rate(small, 1000, s) for s in (1, 2, 4, 6)}
    print("L2 -> SM by 32 KiB stages in flight:", {s: round(r / 1e12, 2) for s, r in by_stages.items()})
    assert by_stages[1] < by_stages[2] < by_stages[6], by_stages
    with pytest.raises(RuntimeError):
        smo.l2_read_probe(small[1:], 1 << 20, 10, torch.zeros(8, dtype=torch.int64, device="cuda"), 1)
