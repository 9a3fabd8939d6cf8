"""The decode kernel's bounded waits: when an internal signal never comes (the testing flag
NVFP4MLA_FLAG_TEST_TIMEOUT withholds one), the kernel gives up after its wait limit, counts the
timeout in the status word, drains its own copies and returns; the context stays usable and the
next call is correct. Nothing here faults, traps or hangs the GPU."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import attention, pack
from tests.gpu_util import assert_close, bf16_dev, decode_inputs

pytestmark = pytest.mark.gpu


def test_withheld_signal_times_out_and_context_recovers():
    case = workloads.small_case(B=1, Q=1, H=32, topk=300, L=(2000,), seed=77)   # 3 tiles in one CTA
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache)
    q, pt, tk, sl = decode_inputs(case)

    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status, max_ctas=1,
                        test_timeout=True)
    torch.cuda.synchronize()
    st = status.cpu().tolist()
    assert st[2] >= 1 and st[0] == 0 and st[1] == 0, st

    status.zero_()
    out, lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status, max_ctas=1)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, "after a timed-out call")


def test_polling_merge_gives_up_when_partials_never_arrive():
    """With results in pinned host memory the merge blocks poll their unit's partial tags. When
    the decode grid gives up (withheld signal), no tag is written: every merge block's bounded
    wait expires and is counted, and the next call (host results again) is correct."""
    case = workloads.small_case(B=1, Q=1, H=32, topk=300, L=(2000,), seed=78)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache)
    q, pt, tk, sl = decode_inputs(case)
    hout = torch.empty((1, 1, 32, 512), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((1, 1, 32), dtype=torch.float32).pin_memory()

    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, out=hout, lse=hlse, dev_status=status,
                        max_ctas=1, test_timeout=True)
    torch.cuda.synchronize()
    st = status.cpu().tolist()
    # the decode CTA's timeout plus one per merge block (4 blocks of 8 heads)
    assert st[2] >= 1 + 4 and st[0] == 0 and st[1] == 0, st

    status.zero_()
    m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, out=hout, lse=hlse, dev_status=status, max_ctas=1)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(hout, hlse, ref_out, ref_lse, "host results after a timed-out call")
