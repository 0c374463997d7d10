"""The no-allocation indexer + selection entry point, csa_index_topk_static.

Callers that cannot hand the library a workspace (their device memory is reserved by another
allocator, or their serving loop must never call cudaMalloc / cudaFree) use this call: it keeps its
temporary buffers in a fixed device array inside the library. Two calls in a row, with different
inputs and row lengths, must give exactly what csa_index_topk gives with a caller workspace; a
request larger than the array is refused before anything runs. The file name makes pytest collect
it last, so a run that stops at the first failure has run every other test before this one.
"""
import numpy as np
import pytest
import torch

import synth
from tests import _harness as Hn

pytestmark = pytest.mark.gpu


def _inputs(rng, B, n_cap, H_idx=64):
    cidx = synth.round_bf16(rng.standard_normal((B, n_cap, 128), dtype=np.float32) / np.float32(np.sqrt(128)))
    q_idx = synth.round_bf16(rng.standard_normal((B, 1, H_idx, 128), dtype=np.float32) / np.float32(np.sqrt(128)))
    w = (rng.standard_normal((B, 1, H_idx)) / np.sqrt(128 * H_idx)).astype(np.float32)
    pos = np.array([[4 * n_cap - 1 - 5 * b] for b in range(B)], np.int64)
    return (torch.from_numpy(pos).cuda(), Hn.dev(q_idx, "bf16"), torch.from_numpy(w).cuda(),
            Hn.dev(cidx, "bf16"))


def test_static_scratch_matches_workspace_call_twice():
    L = Hn.lib()
    rng = np.random.default_rng(7)
    c = L.Config(top_k=512, ratio=4)
    # first call: one CTA per row, scores kept internal; second: rows needing candidate levels,
    # scores returned to the caller
    for B, n_cap, want_scores in ((8, 16384, False), (3, 40000, True)):
        pos, q_idx, w, cidx = _inputs(rng, B, n_cap)
        ref_topk = torch.empty(B, 1, c.top_k, dtype=torch.int32, device="cuda")
        ref_scores = torch.empty(B, 1, n_cap, dtype=torch.float32, device="cuda")
        L.csa_index_topk(c, pos, q_idx, w, cidx, ref_topk, ref_scores)
        got_topk = torch.full((B, 1, c.top_k), -7, dtype=torch.int32, device="cuda")
        got_scores = torch.full((B, 1, n_cap), float("nan"), device="cuda") if want_scores else None
        L.csa_index_topk_static(c, pos, q_idx, w, cidx, got_topk, got_scores)
        torch.cuda.synchronize()
        assert torch.equal(got_topk, ref_topk), f"B={B} n_cap={n_cap}: selections differ"
        if want_scores:
            for b in range(B):
                V = int(pos[b, 0].item() + 1) // 4
                Hn.check_scores(got_scores[b, 0, :V].double().cpu().numpy(),
                                ref_scores[b, 0, :V].double().cpu().numpy(), "bf16", f"static scores b{b}")
    assert L.csa_get_device_status() == 0


@pytest.mark.parametrize("case", ["f32_simt", "bf16_multi_query", "bf16_caller_scores_large"])
def test_static_scratch_other_paths(case):
    """The other indexer paths that can run without a workspace, twice in a row, against
    csa_index_topk: the float32 CUDA-core indexer (the tiny workload's shape), several queries per
    request, and caller-provided scores for a request whose own score buffer would not fit the
    static array (the scratch then holds only what the call uses)."""
    L = Hn.lib()
    rng = np.random.default_rng(len(case))
    for rep in range(2):
        if case == "f32_simt":
            c = L.Config(H=8, H_idx=8, top_k=64, ratio=4, storage="f32")
            B, S, n_cap, H_idx = 2, 1, 512 - 37 * rep, 8
        elif case == "bf16_multi_query":
            c = L.Config(top_k=512, ratio=4)
            B, S, n_cap, H_idx = 2, 3, 6000 + 1000 * rep, 64
        else:
            c = L.Config(top_k=512, ratio=4)
            B, S, n_cap, H_idx = 2, 80, 16384, 64          # 10.5 MB of scores: beyond the array
        st = c.storage
        cidx = rng.standard_normal((B, n_cap, 128), dtype=np.float32) / np.float32(np.sqrt(128))
        q_idx = rng.standard_normal((B, S, H_idx, 128), dtype=np.float32) / np.float32(np.sqrt(128))
        if st == "bf16":
            cidx, q_idx = synth.round_bf16(cidx), synth.round_bf16(q_idx)
        w = (rng.standard_normal((B, S, H_idx)) / np.sqrt(128 * H_idx)).astype(np.float32)
        pos = np.stack([4 * n_cap - 1 - 9 * np.arange(S) - 5 * b for b in range(B)]).astype(np.int64)
        pos_d, q_d, w_d, c_d = (torch.from_numpy(pos).cuda(), Hn.dev(q_idx, st), torch.from_numpy(w).cuda(),
                                Hn.dev(cidx, st))
        ref_topk = torch.empty(B, S, c.top_k, dtype=torch.int32, device="cuda")
        ref_scores = torch.empty(B, S, n_cap, dtype=torch.float32, device="cuda")
        L.csa_index_topk(c, pos_d, q_d, w_d, c_d, ref_topk, ref_scores)
        got_topk = torch.full((B, S, c.top_k), -7, dtype=torch.int32, device="cuda")
        got_scores = torch.full((B, S, n_cap), float("nan"), device="cuda") if case != "f32_simt" else None
        L.csa_index_topk_static(c, pos_d, q_d, w_d, c_d, got_topk, got_scores)
        torch.cuda.synchronize()
        assert torch.equal(got_topk, ref_topk), f"{case} call {rep}: selections differ"
        if got_scores is not None:
            for b in range(B):
                for s_ in range(S):
                    V = int(pos[b, s_] + 1) // 4
                    Hn.check_scores(got_scores[b, s_, :V].double().cpu().numpy(),
                                    ref_scores[b, s_, :V].double().cpu().numpy(), st, f"{case} b{b} s{s_}")
    assert L.csa_get_device_status() == 0


def test_static_scratch_rejects_oversized_request():
    L = Hn.lib()
    c = L.Config(top_k=512, ratio=4)
    B, n_cap = 64, 65536                        # 16 MiB of scores: beyond the fixed array
    pos = torch.zeros(B, 1, dtype=torch.int64, device="cuda")
    q_idx = torch.zeros(B, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(B, 1, 64, device="cuda")
    cidx = torch.zeros(B, n_cap, 128, dtype=torch.bfloat16, device="cuda")
    topk = torch.full((B, 1, 512), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(L.CsaError) as e:
        L.csa_index_topk_static(c, pos, q_idx, w, cidx, topk)
    assert e.value.status == 4 and "static" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(topk == -7)
