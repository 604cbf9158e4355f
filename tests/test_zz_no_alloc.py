"""fa_fwd_varlen_noalloc: the varlen forward with the planning workspace in
the library's static device array instead of caller memory.

Compared with fa_fwd_varlen (caller workspace) on the same inputs, two calls
in a row each, the outputs must be bit-identical (the same kernels run on
the same task list).  Requests whose task list would not fit the array are
rejected before any CUDA call.  This file is collected last so that the
static array is exercised after every other test has run."""
import numpy as np
import pytest

import synthetic


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


FAKE = 0x10000


def test_oversize_request_rejected_before_cuda(fa):
    cap = fa.fa_noalloc_scratch_bytes()
    assert cap == 1 << 20
    # 16 heads: each 256 queries add 16 tasks of 32 bytes -> 2 MiB of records for 2^19 queries
    total_q = 1 << 19
    assert fa.fa_varlen_workspace_size(4, 16, total_q) > cap
    rc = fa.fa_fwd_varlen_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, total_q, total_q, 16, 16, 128, 128,
                                  1, 0.0, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    # empty problems are fine without any pointer
    assert fa.fa_fwd_varlen_noalloc(None, None, None, None, None, None, None, 0, 0, 0, 16, 16, 128, 128, 1, 0.0,
                                    None) == 0


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice(fa):
    torch = pytest.importorskip("torch")

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    cases = [
        synthetic.VarlenWorkload("na1", (300, 1, 0, 513, 129, 700), (400, 1, 5, 513, 0, 350), 8, 2, 128, 128, True,
                                 seed=11),
        synthetic.VarlenWorkload("na2", (1000, 77, 2048), (1000, 77, 2048), 16, 16, 64, 64, False, seed=12),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    for w in cases:
        q, k, v = (dev(a) for a in w.generate())
        cq = torch.tensor(w.cu_seqlens_q, device="cuda")
        ck = torch.tensor(w.cu_seqlens_k, device="cuda")
        ws = torch.empty(fa.fa_varlen_workspace_size(w.batch, w.heads_q, w.total_q), dtype=torch.uint8,
                         device="cuda")
        outs = []
        for call in range(2):
            for noalloc in (False, True):
                o = torch.full(w.shapes["o"], 3.0, dtype=torch.bfloat16, device="cuda")
                lse = torch.full(w.shapes["lse"], 5.0, dtype=torch.float32, device="cuda")
                args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), cq.data_ptr(),
                        ck.data_ptr(), w.batch, w.total_q, w.total_k, w.heads_q, w.heads_kv, w.d_qk, w.d_v,
                        int(w.causal), w.softmax_scale)
                if noalloc:
                    rc = fa.fa_fwd_varlen_noalloc(*args, stream)
                else:
                    rc = fa.fa_fwd_varlen(*args, ws.data_ptr(), ws.numel(), stream)
                assert rc == 0
                torch.cuda.synchronize()
                code, detail = fa.fa_device_status()
                assert code == 0, detail
                outs.append((noalloc, o, lse))
        ref_o, ref_l = outs[0][1], outs[0][2]
        assert torch.isfinite(ref_o.float()).all()
        for noalloc, o, lse in outs[1:]:
            assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), (w.name, noalloc)
