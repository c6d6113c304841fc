"""GPU parity of the FP8 combine (ep_combine_fp8, through the C ABI): expert
outputs as e4m3 codes plus one float32 scale per 128 channels.  Bit-exact
against the oracle's fp32 sequence (coefficient fl32(w * scale), FMA chain in
j order, one bf16 rounding) and within 2^-7 of its fp64 sum."""
import numpy as np
import pytest
import torch

import oracle
import combine_ep_layout_02_gb300 as ep
from combine_ep_layout_02_gb300 import workloads as W

from gpu_helpers import DEV, check_combine, draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _bits(t):
    return W.bf16_bits(t)


def _run_and_compare(wl, what):
    _, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    y_q, y_s = W.fp8_expert_outputs(wl, device=DEV)
    out = ep.combine_fp8(y_q, y_s, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    dst = lay.dst_row.cpu().numpy()
    qh, sh, wh = y_q.cpu().numpy(), y_s.cpu().numpy(), w.cpu().numpy()
    _, ref, absum = oracle.combine_fp8_f64(qh, sh, wh, dst)
    got = _bits(out)
    check_combine(got, ref, absum, what)
    assert np.array_equal(got, oracle.combine_fp8_fp32_seq(qh, sh, wh, dst)), what


@pytest.mark.parametrize("name,T,H", [("small", 128, 2048), ("masked", 2048, 2048),
                                      ("decode_fp8", 600, 7168), ("prefill_fp8", 1100, 1024),
                                      ("prefill", 3000, 384), ("small", 1, 128),
                                      ("decode_fp8", 37, 7168)])
def test_combine_fp8_bit_exact(name, T, H):
    base = W.WORKLOADS[name]
    wl = base.scaled(T=T, H=H, capacity=min(base.capacity, T) or None)
    _run_and_compare(wl, "%s T=%d H=%d" % (name, T, H))


@pytest.mark.parametrize("k,E,H", [(9, 64, 1024), (16, 256, 7168), (32, 1024, 512), (1, 8, 128)])
def test_combine_fp8_topk_beyond_one_batch(k, E, H):
    wl = W.WORKLOADS["small"].scaled(T=300, H=H, k=k, E=E, R=1, expert_out="independent")
    _run_and_compare(wl, "k=%d" % k)


def test_combine_fp8_decodes_every_code():
    # k = 1, weight 1, scale 1: out = bf16(decode(code)), exact for every
    # finite code (e4m3 values are bf16 values); 0x7F and 0xFF give NaN
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(1, 256)
    y_q = codes.repeat(2, 1).to(DEV)
    y_s = torch.ones(2, 2, dtype=torch.float32, device=DEV)
    dst = torch.tensor([[0], [1]], dtype=torch.int32, device=DEV)
    w = torch.ones(2, 1, dtype=torch.float32, device=DEV)
    out = ep.combine_fp8(y_q, y_s, w, dst).cpu()
    expect = codes.view(torch.float8_e4m3fn).float().to(torch.bfloat16)
    nan = (codes == 0x7F) | (codes == 0xFF)
    for row in out:
        assert torch.isnan(row[nan.view(-1)].float()).all()
        finite = ~nan.view(-1)
        got = row[finite].view(torch.int16)
        want = expect.view(-1)[finite].view(torch.int16)
        # the FMA chain starts from +0: code 0x80 (-0) gives +0
        want = torch.where(want == torch.tensor(-32768, dtype=torch.int16), torch.zeros_like(want), want)
        assert torch.equal(got, want)


def test_combine_fp8_dropped_pairs_bad_rows_and_empty_tokens():
    rows, H = 40, 256
    wl = W.WORKLOADS["small"].scaled(T=rows, k=1, H=H)
    y_q, y_s = W.fp8_expert_outputs(wl, device=DEV)
    dst = torch.tensor([[3, -1, 7], [-1, -1, -1], [39, 0, -1], [5, 5, 5], [1, 40, -2]],
                       dtype=torch.int32, device=DEV)
    w = torch.tensor([[0.5, 9.0, 0.25], [1, 1, 1], [1.0, 0.0, 3.0], [1, -1, 0.5], [2, 2, 2]],
                     device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ep.combine_fp8(y_q, y_s, w, dst, status=status)
    assert ep.status_read(status) == ep.EP_FLAG_BAD_ROW            # rows 40 and -2
    dh = dst.cpu().numpy().copy()
    dh[4, 1:] = -1                                                  # what the kernel skipped
    ref = oracle.combine_fp8_fp32_seq(y_q.cpu().numpy(), y_s.cpu().numpy(), w.cpu().numpy(), dh)
    assert np.array_equal(_bits(out), ref)
    assert torch.all(out[1].view(torch.int16) == 0)                 # no valid pair -> +0


def test_combine_fp8_of_dispatched_codes_returns_the_input():
    # dispatch_fp8's own output as the expert outputs (identity experts) and
    # weights summing to ~1: the combine returns x within the e4m3 error
    wl = W.WORKLOADS["decode_fp8"].scaled(T=512, capacity=512)
    x, idx, w = draw(wl, DEV)
    lay = ep.layout(idx, wl.E, wl.R, wl.kind, wl.capacity)
    q, s = ep.dispatch_fp8(x, lay.dst_row, wl.rows, status=lay.status)
    out = ep.combine_fp8(q, s, w, lay.dst_row, status=lay.status)
    assert ep.status_read(lay.status) == 0
    xf = x.double()
    wsum = w.double().sum(1, keepdim=True)
    # every row of a token holds the same codes v ~ x (|v - x| <= 2^-4 |x| in
    # the e4m3 normal range, 2^-10 * scale below it), so the exact sum is
    # v * sum(w); then one bf16 rounding (2^-8 relative) and the fp32 error
    scale = s[lay.dst_row[:, 0].long()].double().repeat_interleave(128, dim=1)
    err_v = (2.0 ** -4 * xf.abs() + 2.0 ** -10 * scale) * wsum
    bound = err_v * (1 + 2.0 ** -7) + 2.0 ** -8 * 1.07 * xf.abs() * wsum
    assert torch.all((out.double() - xf * wsum).abs() <= bound)
