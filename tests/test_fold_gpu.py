"""sparse_mla_decode_shared (query tokens folded over one shared index list) against the oracle:
query token j must equal plain attention over the shared entries whose bit j is set, under the
decode's entry rules (validity, causal range per query token)."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import attention, pack
from tests.gpu_util import assert_close, bf16_dev, i32

pytestmark = pytest.mark.gpu


def _per_query_lists(shared, member, Q):
    """The per-query lists the folded call stands for (entries without bit j become -1)."""
    return np.stack([np.where((member >> j) & 1, shared, -1) for j in range(Q)], axis=1).astype(np.int32)


SPECS = [
    dict(B=2, Q=2, H=16, topk=512, L=(3000, 2600), shared=0.9),          # 2 tokens x 16 heads: one pass
    dict(B=1, Q=4, H=16, topk=512, L=(5000,), shared=0.9),               # 64 columns: two head groups
    dict(B=2, Q=2, H=32, topk=256, L=(2000, 1800), shared=0.5),          # 64 columns, one token per group
    dict(B=2, Q=4, H=32, topk=300, L=(4000, 1900), shared=0.5),          # 128 columns
    dict(B=3, Q=2, H=16, topk=300, L=(1500, 1400, 900), invalid_frac=0.25, dup=True, causal_tail=True),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: "B{B}Q{Q}H{H}K{topk}".format(**s))
@pytest.mark.parametrize("cluster", [None, "any"], ids=["default", "cluster flag (ignored: split)"])
def test_folded_decode_matches_oracle(spec, cluster):
    case = workloads.small_case(seed=200 + len(str(spec)), **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    cache = torch.from_numpy(rows.copy()).cuda()
    shared, member = workloads.fold_lists(case.topk_indices)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = m.sparse_mla_decode_shared(bf16_dev(case.q_bits), cache, i32(case.page_table), i32(shared),
                                          torch.from_numpy(member).cuda(), i32(case.seq_lens), case.softmax_scale,
                                          dev_status=status, cluster=cluster)
    torch.cuda.synchronize()
    lists = _per_query_lists(shared, member, case.Q)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, lists, case.seq_lens,
                                               case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, f"folded {spec}")
    assert status.cpu().tolist()[2] == 0


def test_folded_equals_unfolded_call():
    """The folded call and sparse_mla_decode on the per-query lists it stands for agree within
    the tolerance, for the 2-token x 16-head fold with 90 % shared lists."""
    case = workloads.small_case(B=4, Q=2, H=16, topk=1024, L=(6000, 5000, 7000, 4500), shared=0.9, seed=77)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    cache = torch.from_numpy(rows.copy()).cuda()
    shared, member = workloads.fold_lists(case.topk_indices)
    q, pt, sl = bf16_dev(case.q_bits), i32(case.page_table), i32(case.seq_lens)
    out_f, lse_f = m.sparse_mla_decode_shared(q, cache, pt, i32(shared), torch.from_numpy(member).cuda(), sl,
                                              case.softmax_scale)
    out_u, lse_u = m.sparse_mla_decode(q, cache, pt, i32(case.topk_indices), sl, case.softmax_scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices, case.seq_lens,
                                               case.softmax_scale)
    assert_close(out_f, lse_f, ref_out, ref_lse, "folded")
    assert_close(out_u, lse_u, ref_out, ref_lse, "unfolded")


def test_rejects_unsupported_shapes():
    case = workloads.small_case(B=1, Q=3, H=16, topk=64, L=(500,), seed=5)
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    shared, member = workloads.fold_lists(case.topk_indices)
    with pytest.raises(m.NvFp4MlaError):     # 3 x 16 = 48 heads is not a supported width
        m.sparse_mla_decode_shared(bf16_dev(case.q_bits), cache, i32(case.page_table), i32(shared),
                                   torch.from_numpy(member).cuda(), i32(case.seq_lens), case.softmax_scale)
