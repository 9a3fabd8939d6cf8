"""The pair schedule (NVFP4MLA_FLAG_PAIR): the split decode with the two halves of the 576-wide
contraction in the two CTAs of a 2-CTA cluster, exchanging partial scores every tile.

Its scores, maxima, P and row sums are the split kernel's bit for bit; only PV differs, adding
V.P_hi and V.P_lo in two fp32 accumulators instead of one. So for the same stream-K cut (as many
pairs as split CTAs) its LSE equals the split schedule's bitwise and its outputs agree to within a
bf16 rounding step; it is also checked against the oracle directly, at small sizes and on every
query token of the full-size cases."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import attention, pack
from tests.gpu_util import assert_close, bf16_dev, decode_inputs, oracle_units_from_device_rows

pytestmark = pytest.mark.gpu

SPECS = [
    dict(B=2, Q=1, H=16, topk=200, L=(700, 1000)),                       # ragged tail: 128 + 72
    dict(B=2, Q=1, H=32, topk=300, L=(2000, 900)),
    dict(B=1, Q=4, H=32, topk=256, L=(3000,)),                            # causal across 4 query tokens
    dict(B=3, Q=2, H=64, topk=130, L=(500, 600, 700)),                    # two head groups
    dict(B=1, Q=1, H=128, topk=129, L=(400,)),                            # four head groups
    dict(B=2, Q=2, H=32, topk=384, L=(1500, 1400), invalid_frac=0.25, dup=True, causal_tail=True),
    dict(B=4, Q=1, H=16, topk=50, L=(40, 60, 2000, 64)),                  # short contexts leave -1 entries
    dict(B=1, Q=1, H=32, topk=2048, L=(9000,)),                          # 16 tiles of one unit
    dict(B=6, Q=1, H=32, topk=1000, L=(3000, 1200, 2500, 8000, 900, 4000)),
]


def _spec_id(s):
    return "B{B}Q{Q}H{H}K{topk}".format(**s)


def _setup(spec, seed):
    case = workloads.small_case(seed=seed, **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache)
    return case, rows, cache


def _decode(case, cache, **kw):
    q, pt, tk, sl = decode_inputs(case)
    out, lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def _assert_matches_split(out, lse, out_s, lse_s, what):
    """LSE bitwise; outputs within one bf16 step of the split schedule's (the fp32 sums behind them
    differ only in rounding order)."""
    assert torch.equal(lse, lse_s), f"{what}: lse differs from the split schedule"
    o, os_ = out.float(), out_s.float()
    excess = (o - os_).abs() - (2.0 ** -7 * os_.abs() + 1e-5)
    assert float(excess.max()) <= 0, f"{what}: out differs from the split schedule by {float((o - os_).abs().max()):.3e}"


def _tiles(spec):
    return spec["B"] * spec["Q"] * max(1, spec["H"] // 32) * ((spec["topk"] + 127) // 128)


@pytest.mark.parametrize("spec", SPECS, ids=_spec_id)
def test_plan_reports_pairs(spec):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas, g = m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], cluster="pair")
    pairs = min(sms // 2, _tiles(spec))
    assert (ctas, g) == (2 * pairs, -2)
    ctas, g = m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], max_ctas=3, cluster="pair")
    assert (ctas, g) == (2 * min(3, _tiles(spec)), -2)


@pytest.mark.parametrize("spec", SPECS, ids=_spec_id)
@pytest.mark.parametrize("ranges", [0, 1, 3])
def test_pair_matches_oracle_and_split(spec, ranges):
    case, rows, cache = _setup(spec, 500 + len(str(spec)))
    out, lse = _decode(case, cache, cluster="pair", max_ctas=ranges)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, f"pair {spec} ranges={ranges}")
    n = m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], max_ctas=ranges, cluster="pair")[0] // 2
    out_s, lse_s = _decode(case, cache, max_ctas=n)
    _assert_matches_split(out, lse, out_s, lse_s, f"pair vs split with {n} ranges")
    out2, lse2 = _decode(case, cache, cluster="pair", max_ctas=ranges)    # deterministic across calls
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("cfg", [1, 2, "3s", 4])
def test_pair_full_size_every_unit(cfg):
    """Full-size cases in the pair schedule: every query token against the oracle, and the whole
    output against the split schedule cut into as many ranges."""
    case = workloads.make_case(cfg)
    rows_total = case.num_pages * 64
    lat, rope = workloads.device_rows(case, rows_total, "cuda")
    cache = torch.empty((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(lat, rope, torch.arange(rows_total, device="cuda"), cache)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = _decode(case, cache, dev_status=status, cluster="pair")
    assert status.cpu().tolist() == [0, 0, 0, 0]
    n = m.sparse_mla_decode_plan(case.B, case.Q, case.H, case.topk, cluster="pair")[0] // 2
    out_s, lse_s = _decode(case, cache, max_ctas=n)
    _assert_matches_split(out, lse, out_s, lse_s, f"pair cfg {cfg}")
    units = [(b, j) for b in range(case.B) for j in range(case.Q)]
    ref = oracle_units_from_device_rows(case, units, lat, rope)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for (b, j), (ro, rl) in ref.items():
        assert_close(o[b, j], l[b, j], ro, rl, f"pair cfg {cfg} unit {(b, j)}")


def test_pair_withheld_signal_times_out_and_context_recovers():
    """Both CTAs of the pair give up on their bounded waits (the producers withhold tile 1's row
    table), count it, drain their copies, meet at the closing cluster barrier and return; the
    next call is correct."""
    spec = dict(B=1, Q=1, H=32, topk=300, L=(2000,))
    case, rows, cache = _setup(spec, 79)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    _decode(case, cache, dev_status=status, cluster="pair", max_ctas=1, test_timeout=True)
    st = status.cpu().tolist()
    assert st[2] >= 1 and st[0] == 0 and st[1] == 0, st
    status.zero_()
    out, lse = _decode(case, cache, dev_status=status, cluster="pair", max_ctas=1)
    assert status.cpu().tolist() == [0, 0, 0, 0]
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, "pair after a timed-out call")
