"""The backward entry point that allocates nothing.

lsr_replay_attn_bwd_noalloc is for callers that cannot allocate device
memory where they run the backward (no cudaMalloc/cudaFree allowed there,
or a plain C caller without a device allocator).  It uses the library's
built-in 64 MiB scratch instead of a caller workspace.  These tests call it
through the C ABI twice in a row, on blocks of different sizes so that the
second call starts from the first call's leftover scratch, and compare each
result with lsr_replay_attn_bwd given its own workspace and with the fp64
oracle, within the gradient tolerance of the other parity tests.  The
second block has more shards than prompt pages, so some dQ slices cover no
keys at all and must be written as zeros over the first call's leftovers.
This file is collected last so that a run stopping at the first failure
has run every other test.
"""
import pytest
import torch

import oracle
from helpers import GRAD_RELL2, lib, rel_l2
from resident_prefix_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _block(cfg, seed):
    L = lib()
    from resident_prefix_attention_gb300.replay import ReplaySession
    wl = W.make_workload(cfg, seed=seed)
    resp = wl.responses[0]
    sess = ReplaySession(wl.page_table.numel(), cfg.Hkv, cfg.page_size, cfg.d,
                         wl.page_table)
    sess.write(wl.k_prompt.cuda(), wl.v_prompt.cuda(), 0)
    sess.write(resp.k.cuda(), resp.v.cuda(), cfg.P)
    q, dO = resp.q.cuda(), resp.dO.cuda()
    res = sess.forward_block(q, cfg.P, 0, cfg.shards, cfg.scale)
    return L, sess, q, dO, res


def _grads(sess, q, cfg):
    dq = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    dk, dv = sess.grad_pages(cfg.R)
    return dq, dk, dv


def _logical(pages, R, Hkv, d):
    """Logical [R, Hkv, d] view of response gradient pages."""
    n, _, ps, _ = pages.shape
    return pages.permute(0, 2, 1, 3).reshape(n * ps, Hkv, d)[:R]


def test_noalloc_backward_matches_workspace_backward_twice():
    cases = [
        # 8 prompt pages in 4 shards: every half-shard holds one page
        W.make_config("mid", name="noalloc-a", P=2048, R=300, shards=4),
        # 4 prompt pages in 6 shards: two shards and four half-shards are
        # empty, so their dQ slices are zero-filled over leftover scratch
        W.make_config("mid", name="noalloc-b", P=1024, R=200, shards=6),
    ]
    runs = [(cfg,) + _block(cfg, seed) for seed, cfg in enumerate(cases)]
    for seed, (cfg, L, sess, q, dO, res) in enumerate(runs):  # in a row
        ref = _grads(sess, q, cfg)
        n = L.lsr_bwd_workspace_size(cfg.shards, cfg.Hq, cfg.R, cfg.d)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        L.lsr_replay_attn_bwd(sess.pool, q, res.o, dO, res.lse, cfg.P, 0,
                              sess.page_table, cfg.shards, cfg.scale, *ref, ws)
        got = _grads(sess, q, cfg)
        L.lsr_replay_attn_bwd_noalloc(sess.pool, q, res.o, dO, res.lse, cfg.P,
                                      0, sess.page_table, cfg.shards,
                                      cfg.scale, *got)
        torch.cuda.synchronize()
        assert sess.device_status() == 0
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            e = rel_l2(a, b)
            assert e <= GRAD_RELL2, f"{cfg.name} {name} rel-L2 {e:.3e}"
        wl = W.make_workload(cfg, seed=seed)
        resp = wl.responses[0]
        want = oracle.attention_backward(resp.q, wl.k_prompt, wl.v_prompt,
                                         resp.k, resp.v, resp.dO, 0,
                                         cfg.scale)
        mine = (got[0], _logical(got[1], cfg.R, cfg.Hkv, cfg.d),
                _logical(got[2], cfg.R, cfg.Hkv, cfg.d))
        for name, a, b in zip(("dq", "dk", "dv"), mine, want):
            e = rel_l2(a, b)
            assert e <= GRAD_RELL2, f"{cfg.name} {name} vs oracle {e:.3e}"


def test_noalloc_rejects_blocks_beyond_its_scratch():
    cfg = W.make_config("mid", name="noalloc-big", P=1024, R=4096, shards=1)
    L, sess, q, dO, res = _block(cfg, 5)
    # 2*shards+1 = 3 dQ slices x 4096 rows x 32 heads x 128 x 4 bytes
    # = 192 MiB, plus D, against the 64 MiB scratch
    assert (L.lsr_bwd_workspace_size(cfg.shards, cfg.Hq, cfg.R, cfg.d)
            > 64 * 2 ** 20)
    dq, dk, dv = _grads(sess, q, cfg)
    with pytest.raises(L.LsrError) as err:
        L.lsr_replay_attn_bwd_noalloc(sess.pool, q, res.o, dO, res.lse, cfg.P,
                                      0, sess.page_table, cfg.shards,
                                      cfg.scale, dq, dk, dv)
    assert err.value.status == L.LSR_ERR_INVALID_ARG
    assert "64 MiB" in str(err.value)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dq) == 0 and torch.count_nonzero(dk) == 0
