"""sparse_mla_decode against the oracle on score distributions the synthetic workloads never
reach: one dominant token with every other score a fixed number of log2 units below it (the
regime where 16-bit softmax weights can underflow), a dominant minimum, all-equal scores, and
queries whose elements span a very wide dynamic range.

The pages run the kernel with FP16 operands and FP32 accumulation ("Prime Inference: serving
GLM-5.3 to agents is a KV-cache problem", "A kernel that reads four bits directly"); these
cases check that the rounding of the softmax weights to a 16-bit type does not lose mass that
the tolerance would notice."""
import math

import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import attention, pack
from tests.gpu_util import assert_close, bf16_dev, decode_inputs

pytestmark = pytest.mark.gpu

L = 4096
K = 2048
H = 32
# log2-unit gaps between the dominant score and all the others, one per head (the last
# heads use negative gaps: the "dominant" token is then far below all the others)
GAPS = [17, 20, 24, 10, 15, 16, 18, 19, 21, 22, 23, 25, 26, 28, 30, 40,
        0.5, 1, 2, 4, 8, 12, 14, 33, 36, 60, -17, -24, -10, -30, 0, 5]


def _bf16(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _phys(case, pos):
    return int(case.page_table[0][pos // 64]) * 64 + pos % 64


def _case_with_dominant(where: str, seed: int):
    case = workloads.small_case(B=1, Q=1, H=H, topk=K, L=(L,), seed=seed)
    rng = np.random.default_rng(seed)
    idx = rng.permutation(L)[:K].astype(np.int32)
    dom_pos = int(idx[0])
    slot = {"first": 0, "last": K - 1, "middle": K // 2 + 37}[where]
    idx[0], idx[slot] = idx[slot], idx[0]
    case.topk_indices = idx.reshape(1, 1, K)
    rows = case.num_pages * 64
    lat = np.zeros((rows, 512), np.float32)
    rope = np.zeros((rows, 64), np.float32)
    # every other token: latent dims 16..31 = 6 (block scale 1, exact), score 0
    lat[:, 16:32] = 6.0
    # the dominant token: latent dim 0 = 6 (exact), dims 16..31 = 0
    d = _phys(case, dom_pos)
    lat[d, 16:32] = 0.0
    lat[d, 0] = 6.0
    # q: only dim 0 is non-zero, a_h chosen so that the dominant score sits GAPS[h] log2 units
    # above the others (z_d - z_o = scale * a * 6 = gap * ln 2)
    q = np.zeros((1, 1, H, 576), np.float32)
    for h, gap in enumerate(GAPS):
        q[0, 0, h, 0] = gap * math.log(2.0) / (6.0 * case.softmax_scale)
    case.q_bits = _bf16(q)
    return case, _bf16(lat), _bf16(rope)


def _run(case, lat, rope):
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache)
    q, pt, tk, sl = decode_inputs(case)
    out, lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale)
    torch.cuda.synchronize()
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    return out, lse, ref_out, ref_lse


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_dominant_token_with_others_far_below(where):
    case, lat, rope = _case_with_dominant(where, seed=70 + len(where))
    out, lse, ref_out, ref_lse = _run(case, lat, rope)
    # the mass of the 2,047 others is visible in dims 16..31 of the reference (e.g. 1.5 % of
    # the weight at a 17-unit gap): it must be visible in the kernel's output too
    assert ref_out[0, 0, 0, 16] > 0.05
    assert_close(out, lse, ref_out, ref_lse, f"dominant {where}")


def test_all_scores_equal():
    case = workloads.small_case(B=1, Q=1, H=H, topk=K, L=(L,), seed=81)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    case.q_bits[:] = 0
    out, lse, ref_out, ref_lse = _run(case, lat, rope)
    np.testing.assert_allclose(ref_lse[0, 0], math.log(K), atol=1e-12)
    assert_close(out, lse, ref_out, ref_lse, "all scores equal")


def test_query_with_wide_dynamic_range():
    """q elements log-uniform in magnitude from 2^-30 to 2^3 of the largest one (random signs)
    for half the heads; the rest of the case is a standard random case."""
    case = workloads.small_case(B=2, Q=1, H=H, topk=700, L=(3000, 2500), seed=83)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rng = np.random.default_rng(84)
    q = np.zeros((2, 1, H, 576), np.float32)
    q[:] = rng.standard_normal(q.shape).astype(np.float32)
    e = rng.uniform(-30.0, 3.0, size=(2, 1, H // 2, 576))
    sgn = np.where(rng.random(e.shape) < 0.5, -1.0, 1.0)
    q[:, :, : H // 2, :] = (sgn * np.exp2(e)).astype(np.float32)
    case.q_bits = _bf16(q)
    out, lse, ref_out, ref_lse = _run(case, lat, rope)
    assert_close(out, lse, ref_out, ref_lse, "wide q range")
