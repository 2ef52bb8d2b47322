"""page_score_topk_static_scratch: the scoring call for callers that cannot
allocate device memory (an engine whose pool allocator already owns all of
HBM, a runtime without a device-allocation hook, a decode loop that must not
take cudaMalloc's device synchronisation).  It uses the library's fixed device
scratch instead of a caller workspace, and must give exactly what
page_score_topk gives, call after call, even though every call reuses the
same scratch.

This file is collected last on purpose, so a run that stops at its first
failure has already run every other test; it also passes on its own.
"""
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from paged_kv_cache_minmax_gb300 import build

    build.build_library()
    kvmm.load()
    oracle.build()


def test_static_scratch_scoring_matches_workspace_scoring_twice():
    cfg = workloads.scaled(workloads.CONFIGS[2], B=2, L=2, S=4096 + 9, K=32, n_planted=16, ragged=True)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    s = st.shape
    mask = torch.ones(cfg.L, cfg.Hkv, dtype=torch.uint8, device="cuda")
    mask[1, 3] = 0  # one unit keeps its previous selection in both paths
    for call, layer in enumerate((0, 1)):
        q = wl.q[layer] if call == 0 else (wl.q[layer].float() * -0.5).to(torch.bfloat16)
        ref_idx = torch.full_like(st.sel_idx, -7)
        ref_cnt = torch.full_like(st.sel_cnt, -7)
        got_idx = ref_idx.clone()
        got_cnt = ref_cnt.clone()
        ref_sc = torch.zeros(cfg.B, cfg.Hkv, cfg.Pmax, device="cuda")
        got_sc = torch.zeros_like(ref_sc)
        kvmm.page_score_topk(s, layer, q, st.meta, wl.seq_len, mask, cfg.K, ref_idx, ref_cnt, st.workspace,
                             st.err, scores_out=ref_sc)
        kvmm.page_score_topk_static_scratch(s, layer, q, st.meta, wl.seq_len, mask, cfg.K, got_idx, got_cnt,
                                            st.err, scores_out=got_sc)
        torch.cuda.synchronize()
        assert st.read_err() == 0
        assert torch.equal(got_cnt, ref_cnt), f"call {call}: counts differ"
        assert torch.equal(got_idx, ref_idx), f"call {call}: selections differ"
        # the same kernels on the same inputs: the scores agree bit for bit
        assert torch.equal(got_sc, ref_sc), f"call {call}: scores differ"
        assert int(got_cnt[0, layer, 0]) == cfg.K
        # and against the oracle: scores within tolerance, the selection the top K of its own scores and the
        # oracle's up to counted ties
        stats = parity.Stats()
        for b, h in ((0, 0), (cfg.B - 1, cfg.Hkv - 1)):
            if not mask[layer, h]:
                continue
            seq = int(wl.seq_len[b])
            P = -(-seq // cfg.T)
            kp, _, row = parity.unit_pool(wl, b, layer, h)
            meta_o, _ = oracle.unit_minmax(kp, cfg.T, row, seq)
            s_o = oracle.unit_scores(parity.q_group(wl, q, b, h), meta_o, P, 0)
            sel = got_idx[b, layer, h, : int(got_cnt[b, layer, h])].cpu().numpy()
            parity.check_selection(got_sc[b, h, :P].double().cpu().numpy(), s_o, sel, cfg.K, stats)


def test_static_scratch_rejects_shapes_beyond_its_size():
    # 8 * 8 units * 32768 pages of scores is 8 MiB, beyond the 4 MiB scratch: rejected before any launch
    s = kvmm.make_shape(8, 1, 32, 8, 128, 16, 32768, 128, 8 * 8 * 32768)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    bf = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    status = kvmm.load().page_score_topk_static_scratch(
        kvmm.ctypes.byref(s), 0, bf.data_ptr(), bf.data_ptr(), dummy.data_ptr(), None, 8, 0, dummy.data_ptr(),
        dummy.data_ptr(), None, None, torch.cuda.current_stream().cuda_stream)
    assert status == kvmm.WORKSPACE_TOO_SMALL
