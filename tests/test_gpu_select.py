"""Selection, gather and page-table kernels alone, on seeded inputs: bit-exact against the oracle."""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth as S
from oracle import kvsel_oracle as O

pytestmark = pytest.mark.gpu


def _ws(K, desc, cuda):
    n = K.kvsel_workspace_size(desc)
    buf = torch.zeros(n + K.WS_ALIGN, dtype=torch.uint8, device=cuda)
    off = (-buf.data_ptr()) % K.WS_ALIGN
    return buf[off:off + n]


@pytest.mark.parametrize("rows,n,k,ties", [(3, 100, 7, True), (5, 4097, 1000, True), (2, 33000, 1024, False),
                                           (2, 50000, 4096, True), (4, 300, 300, True), (2, 64, 0, False),
                                           (3, 70000, 1, True),
                                           # more rows than one wave of 512-thread CTAs: the 256-thread kernels
                                           (400, 3000, 200, True), (330, 16384, 1024, True)])
def test_topk_token_mode_exact(rows, n, k, ties, cuda):
    """Top-k with ties to the lower index, both decided in fp32 (the kernel's precision)."""
    from attention_kv_cache_gb300 import kvsel as K
    W = 3
    s = S.random_scores(rows, n, seed=rows * 1000 + n, ties=ties)
    desc = K.make_desc(n_layers=rows, h_q=1, h_kv=1, head_dim=128, window=W, prefix_lens=[n])
    idx = torch.full((rows, k + W), -7, dtype=torch.int32, device=cuda)
    ws = _ws(K, desc, cuda)
    K.kvsel_topk(desc, s.to(cuda), rows, k, 0, idx, ws)
    got = idx.cpu().numpy()
    for r in range(rows):
        want = O.select_tokens(s[r].double().numpy(), k, n, W)
        np.testing.assert_array_equal(got[r], want)


@pytest.mark.parametrize("L,P,k,n_recent,W", [(8192, 16, 128, 4, 32), (8200, 16, 50, 1, 16), (1000, 8, 3, 2, 8),
                                               (131072, 16, 128, 4, 32)])
def test_topk_page_mode_exact(L, P, k, n_recent, W, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    n_pages = -(-L // P)
    rows = 3
    s = S.random_scores(rows, n_pages, seed=L + P, ties=True)
    desc = K.make_desc(n_layers=rows, h_q=1, h_kv=1, head_dim=128, window=W, prefix_lens=[L], page_size=P)
    n_sel = k + n_recent + W // P
    idx = torch.full((rows, n_sel), -7, dtype=torch.int32, device=cuda)
    K.kvsel_topk(desc, s.to(cuda), rows, k, n_recent, idx, _ws(K, desc, cuda))
    got = idx.cpu().numpy()
    for r in range(rows):
        want = O.select_pages(s[r].double().numpy(), k, n_recent, L, W, P)
        np.testing.assert_array_equal(got[r], want)


@pytest.mark.parametrize("P", [1, 16])
def test_compact_bit_exact_and_bounds(P, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    w = S.Workload("gather", 95, 3, 4, 2, 128, 16, (999,), k_keep=20, page_size=P, n_recent=1 if P > 1 else 0)
    inp = S.make_inputs(w, "cpu")
    n_keys = 999 + 16
    lim = n_keys if P == 1 else -(-n_keys // P)
    g = torch.Generator().manual_seed(3)
    n_sel = 23
    idx = torch.randint(0, lim, (1, w.n_layers, w.h_kv, n_sel), generator=g, dtype=torch.int32)
    desc = K.make_desc(n_layers=w.n_layers, h_q=w.h_q, h_kv=w.h_kv, head_dim=128, window=16, prefix_lens=[999],
                       page_size=P)
    kd, vd = inp.k[0].to(cuda), inp.v[0].to(cuda)
    ko = torch.empty((1, w.n_layers, w.h_kv, n_sel * P, 128), dtype=torch.bfloat16, device=cuda)
    vo = torch.empty_like(ko)
    ws = _ws(K, desc, cuda)
    K.kvsel_compact(desc, kd, vd, idx.to(cuda), w.n_layers, n_sel, ko, vo, ws)
    assert K.kvsel_read_device_error(ws) == K.OK
    for layer in range(w.n_layers):
        for h in range(w.h_kv):
            want_k = O.gather_rows(inp.k[0][layer, h].float().numpy(), idx[0, layer, h].numpy().astype(np.int64), P)
            want_v = O.gather_rows(inp.v[0][layer, h].float().numpy(), idx[0, layer, h].numpy().astype(np.int64), P)
            np.testing.assert_array_equal(ko[0, layer, h].float().cpu().numpy(), want_k)
            np.testing.assert_array_equal(vo[0, layer, h].float().cpu().numpy(), want_v)
    # an index out of range is not followed: its rows are zero and the error word says so
    bad = idx.clone()
    bad[0, 1, 0, 5] = lim
    bad[0, 2, 1, 0] = -1
    K.kvsel_compact(desc, kd, vd, bad.to(cuda), w.n_layers, n_sel, ko, vo, ws)
    assert K.kvsel_read_device_error(ws) == K.ERR_DEVICE
    assert K.kvsel_read_device_error(ws) == K.OK            # reading clears it
    assert torch.all(ko[0, 1, 0, 5 * P:6 * P] == 0) and torch.all(ko[0, 2, 1, 0:P] == 0)


@pytest.mark.parametrize("P", [1, 16])
def test_compact_from_pinned_host_memory(P, cuda):
    """K and V in mapped pinned host memory: the gather reads the kept rows over the host link and
    writes exactly what it writes from device memory; pageable memory is refused before any launch."""
    from attention_kv_cache_gb300 import kvsel as K
    w = S.Workload("gather_host", 96, 3, 4, 2, 128, 16, (2000,), k_keep=20, page_size=P, n_recent=1 if P > 1 else 0)
    inp = S.make_inputs(w, "cpu")
    n_keys = 2000 + 16
    lim = n_keys if P == 1 else -(-n_keys // P)
    n_sel = 37
    idx = torch.randint(0, lim, (1, w.n_layers, w.h_kv, n_sel), generator=torch.Generator().manual_seed(5),
                        dtype=torch.int32).to(cuda)
    desc = K.make_desc(n_layers=w.n_layers, h_q=w.h_q, h_kv=w.h_kv, head_dim=128, window=16, prefix_lens=[2000],
                       page_size=P)
    kd, vd = inp.k[0].to(cuda), inp.v[0].to(cuda)
    kh, vh = inp.k[0].contiguous().pin_memory(), inp.v[0].contiguous().pin_memory()
    ws = _ws(K, desc, cuda)
    out = lambda: torch.full((1, w.n_layers, w.h_kv, n_sel * P, 128), 7.0, dtype=torch.bfloat16, device=cuda)
    ko, vo, ko2, vo2 = out(), out(), out(), out()
    K.kvsel_compact(desc, kd, vd, idx, w.n_layers, n_sel, ko, vo, ws)
    K.kvsel_compact(desc, kd, vh, idx, w.n_layers, n_sel, ko2, vo2, ws)         # V on the host
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    assert torch.equal(ko, ko2) and torch.equal(vo, vo2)
    K.kvsel_compact(desc, kh, vh, idx, w.n_layers, n_sel, ko2, vo2, ws)         # both on the host
    assert K.kvsel_read_device_error(ws) == K.OK
    assert torch.equal(ko, ko2) and torch.equal(vo, vo2)
    pageable = inp.v[0].contiguous()
    assert not pageable.is_pinned()
    n0 = K.kvsel_launch_count()
    with pytest.raises(K.KvselError) as e:
        K.kvsel_compact(desc, kd, pageable, idx, w.n_layers, n_sel, ko2, vo2, ws)
    assert e.value.status == K.ERR_INVALID_ARG and K.kvsel_launch_count() == n0


def test_pagetable_full_size_ragged(cuda):
    """Block union over the ragged batch's full mask (8 sequences, 32 layers, 16 Q blocks)."""
    from attention_kv_cache_gb300 import kvsel as K
    w = S.RAGGED_B8
    M, n_kv = S.block_mask(w, "cpu")
    desc = K.make_desc(n_layers=w.n_layers, h_q=w.h_q, h_kv=w.h_kv, head_dim=128, window=w.window,
                       prefix_lens=w.prefix_lens)
    rows = w.batch * w.n_layers * w.h_kv
    nmax = M.shape[-1]
    indptr = torch.empty(rows + 1, dtype=torch.int32, device=cuda)
    indices = torch.full((rows * nmax,), -1, dtype=torch.int32, device=cuda)
    K.kvsel_pagetable(desc, M.to(cuda), M.shape[3], nmax, n_kv, indptr, indices, _ws(K, desc, cuda))
    ref_ptr, ref_idx = O.block_union_csr(M.numpy(), w.h_kv, n_kv)
    np.testing.assert_array_equal(indptr.cpu().numpy(), ref_ptr)
    np.testing.assert_array_equal(indices.cpu().numpy()[: ref_ptr[-1]], ref_idx)
    density = M.float().mean().item()
    assert 0.05 < density < 0.2


def test_bounded_wait_reports_timeout(cuda):
    """A device wait that nothing completes gives up and reports KVSEL_ERR_TIMEOUT; the context stays usable."""
    from attention_kv_cache_gb300 import kvsel as K
    desc = K.make_desc(n_layers=1, h_q=4, h_kv=2, head_dim=64, window=16, prefix_lens=[512])
    ws = _ws(K, desc, cuda)
    K.kvsel_selftest_bounded_wait(ws, 2000, arrive=False)
    assert K.kvsel_read_device_error(ws) == K.ERR_TIMEOUT
    K.kvsel_selftest_bounded_wait(ws, 2000, arrive=True)
    assert K.kvsel_read_device_error(ws) == K.OK
    # the device still computes after the timeout
    s = S.random_scores(2, 300, seed=5, ties=True)
    idx = torch.empty((2, 10 + 16), dtype=torch.int32, device=cuda)
    d2 = K.make_desc(n_layers=2, h_q=1, h_kv=1, head_dim=64, window=16, prefix_lens=[300])
    K.kvsel_topk(d2, s.to(cuda), 2, 10, 0, idx, _ws(K, d2, cuda))
    for r in range(2):
        np.testing.assert_array_equal(idx[r].cpu().numpy(), O.select_tokens(s[r].double().numpy(), 10, 300, 16))


def test_topk_first_call_in_fresh_process(cuda):
    """The first top-k launch of a process, on rows whose keys fit shared memory, launches (the kernel's
    static shared memory counts against the default limit too)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys, torch; sys.path.insert(0, %r)\n"
        "from attention_kv_cache_gb300 import kvsel as K\n"
        "d = K.make_desc(n_layers=1, h_q=1, h_kv=1, head_dim=128, window=8, prefix_lens=[8192])\n"
        "n = K.kvsel_workspace_size(d); ws = torch.zeros(n + 256, dtype=torch.uint8, device='cuda')\n"
        "ws = ws[(-ws.data_ptr()) %% 256:][:n]\n"
        "s = torch.rand(8192, device='cuda'); idx = torch.empty(18, dtype=torch.int32, device='cuda')\n"
        "K.kvsel_topk(d, s, 1, 10, 0, idx, ws); torch.cuda.synchronize()\n"
        "ref = torch.sort(torch.topk(s, 10).indices).values.int()\n"
        "assert torch.equal(idx[:10], ref), (idx, ref)\n"
        "print('ok')\n" % root)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stderr[-2000:]


@pytest.mark.parametrize("pattern", ["smooth", "top_on_sample_grid", "top_off_sample_grid", "ties_at_threshold",
                                     "top_in_one_segment",
                                     "long_row_global"])
def test_topk_candidate_path_exact(pattern, cuda):
    """Rows long enough for the sampled threshold: the candidate list (smooth scores; the top keys
    never sampled; ties around the k-th key) and the fall-back to the whole-row select (the top keys
    all on the sample's positions, so the threshold keeps fewer than k keys), bit-exact."""
    from attention_kv_cache_gb300 import kvsel as K
    rows, W = 3, 4
    n, k = (65536, 4096) if pattern == "long_row_global" else (32768, 1024)
    g = torch.Generator().manual_seed(77 + len(pattern))
    s = torch.rand((rows, n), generator=g, dtype=torch.float64) ** 8
    stride = n // 1024                                   # the sample's positions are multiples of n / 1024
    if pattern == "top_on_sample_grid":
        s[:, ::stride] += 10.0
    elif pattern == "top_off_sample_grid":
        s[:, 1::stride] += 10.0
    elif pattern == "ties_at_threshold":
        s = torch.round(s * 512) / 512
    elif pattern == "top_in_one_segment":                # one warp's segment holds a third of the
        s[:, :600] += 10.0                               # candidates: its placement offsets dominate
    s = s.float()
    desc = K.make_desc(n_layers=rows, h_q=1, h_kv=1, head_dim=128, window=W, prefix_lens=[n])
    idx = torch.full((rows, k + W), -7, dtype=torch.int32, device=cuda)
    K.kvsel_topk(desc, s.to(cuda), rows, k, 0, idx, _ws(K, desc, cuda))
    got = idx.cpu().numpy()
    for r in range(rows):
        np.testing.assert_array_equal(got[r], O.select_tokens(s[r].double().numpy(), k, n, W), err_msg=f"row {r}")
