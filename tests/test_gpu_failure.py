"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes must give up, report through the device status word, and leave the
context usable for the next call.  The attention kernels' own abort path is
exercised the same way: their pipeline waits get a limit short enough to run
out in the ordinary course of a replay, and every CTA that gives up must
drain its copies and products, free its tensor memory and exit cleanly."""
import pytest
import torch

from helpers import lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    L = lib()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    L.lsr_selftest_bounded_wait(status, 2000)      # 2 ms limit
    torch.cuda.synchronize()
    assert int(status[0]) & L.LSR_DEV_WAIT_TIMEOUT
    # the context still works: a page write afterwards is exact
    kp = torch.zeros(2, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    pool = L.lsr_page_pool_create(kp, vp, st)
    k = torch.randn(64, 1, 64, device="cuda").to(torch.bfloat16)
    table = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    L.lsr_write_prefix_pages(pool, k, k, 0, table)
    torch.cuda.synchronize()
    assert torch.equal(kp[1, 0], k[:, 0])
    assert L.lsr_pool_device_status(pool) == 0


def test_selftest_rejects_bad_limits():
    L = lib()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(L.LsrError):
        L.lsr_selftest_bounded_wait(status, 0)


def _kv_replay(sess, wl, cfg, blocks):
    dev = sess.device
    resp = wl.responses[0]
    q, dO = resp.q.to(dev), resp.dO.to(dev)
    dq = torch.zeros(q.shape, dtype=torch.float32, device=dev)
    dk, dv = sess.grad_pages(cfg.R)
    o, lse = sess.replay_response(q, dO, cfg.P, blocks, cfg.shards,
                                  cfg.scale, dq, dk, dv)
    torch.cuda.synchronize()
    n = dk.shape[0]
    gk = dk.permute(0, 2, 1, 3).reshape(n * cfg.page_size, cfg.Hkv,
                                        cfg.d)[:cfg.R]
    gv = dv.permute(0, 2, 1, 3).reshape(n * cfg.page_size, cfg.Hkv,
                                        cfg.d)[:cfg.R]
    return o, lse, dq, gk, gv


def test_attention_kernels_abort_when_a_pipeline_wait_runs_out():
    """With a pipeline wait limit of 1 microsecond the forward, dQ and dK/dV
    kernels' waits run out in the ordinary course of a replay (no role
    stalls on purpose).  A CTA whose wait runs out sets
    LSR_DEV_WAIT_TIMEOUT, lets its issued copies and products finish, frees
    its tensor memory and exits.  Nothing faults, and the next replay on
    the same pool with the default limit matches the oracle."""
    L = lib()
    import oracle
    from helpers import (GRAD_RELL2, LSE_MAXABS, O_MAXABS, max_abs,
                         rel_l2)
    from resident_prefix_attention_gb300 import workloads as W
    from resident_prefix_attention_gb300.replay import ReplaySession
    cfg = W.make_config("mid", name="abort", P=8192, R=512, shards=4)
    wl = W.make_workload(cfg, seed=21)
    resp = wl.responses[0]
    sess = ReplaySession(wl.page_table.numel(), cfg.Hkv, cfg.page_size,
                         cfg.d, wl.page_table)
    dev = sess.device
    sess.write(wl.k_prompt.to(dev), wl.v_prompt.to(dev), 0)
    sess.write(resp.k.to(dev), resp.v.to(dev), cfg.P)
    torch.cuda.synchronize()
    L.lsr_pool_set_wait_limit(sess.pool, 1)
    _kv_replay(sess, wl, cfg, 2)
    status = int(sess.status[0])
    assert status & L.LSR_DEV_WAIT_TIMEOUT, hex(status)
    assert status & ~L.LSR_DEV_WAIT_TIMEOUT == 0, hex(status)
    # default limit again, status cleared: the pool works and is exact
    L.lsr_pool_set_wait_limit(sess.pool, 0)
    sess.status.zero_()
    o, lse, dq, gk, gv = _kv_replay(sess, wl, cfg, 2)
    assert sess.device_status() == 0
    O, lse_ref, dq_ref, dk_ref, dv_ref = oracle.reverse_block_replay(
        resp.q, wl.k_prompt, wl.v_prompt, resp.k, resp.v, resp.dO, 2,
        cfg.scale)
    assert max_abs(o, O) <= O_MAXABS
    assert max_abs(lse, lse_ref) <= LSE_MAXABS
    for x, r in ((dq, dq_ref), (gk, dk_ref), (gv, dv_ref)):
        assert rel_l2(x, r) <= GRAD_RELL2


def test_latent_kernels_abort_when_a_pipeline_wait_runs_out():
    """The same on latent pages: the latent forward, dq~ and latent-row
    kernels give up cleanly under a 1 microsecond wait limit, and the next
    replay with the default limit matches the latent oracle."""
    L = lib()
    import oracle.latent as OL
    from helpers import GRAD_RELL2, LSE_MAXABS, O_MAXABS, max_abs, rel_l2
    from resident_prefix_attention_gb300 import workloads as W
    from resident_prefix_attention_gb300.replay import LatentReplaySession
    cfg = W.make_latent_config("latent_mid", name="abort_latent", P=4096,
                               R=256, shards=4, blocks=1)
    wl = W.make_latent_workload(cfg, seed=22)
    sess = LatentReplaySession(wl.page_table.numel(), cfg.page_size,
                               wl.page_table, cfg.d_c, cfg.d_r)
    dev = sess.device
    sess.write(wl.lat_prompt.to(dev), 0)
    sess.write(wl.lat_resp.to(dev), cfg.P)
    q, dO = wl.q.to(dev), wl.dO.to(dev)

    def replay():
        dq = torch.zeros(q.shape, dtype=torch.float32, device=dev)
        dlat = sess.grad_pages(cfg.R)
        o, lse = sess.replay_response(q, dO, cfg.P, 1, cfg.shards, cfg.scale,
                                      dq, dlat)
        torch.cuda.synchronize()
        return o, lse, dq, dlat

    L.lsr_pool_set_wait_limit(sess.pool, 1)
    replay()
    status = int(sess.status[0])
    assert status & L.LSR_DEV_WAIT_TIMEOUT, hex(status)
    assert status & ~L.LSR_DEV_WAIT_TIMEOUT == 0, hex(status)
    L.lsr_pool_set_wait_limit(sess.pool, 0)
    sess.status.zero_()
    o, lse, dq, dlat = replay()
    assert sess.device_status() == 0
    O, lse_ref = OL.latent_forward(wl.q, wl.lat_prompt, wl.lat_resp, 0,
                                   cfg.scale, cfg.d_c)
    dq_ref, dl_ref = OL.latent_backward(wl.q, wl.lat_prompt, wl.lat_resp,
                                        wl.dO, 0, cfg.scale, cfg.d_c)
    assert max_abs(o, O) <= O_MAXABS
    assert max_abs(lse, lse_ref) <= LSE_MAXABS
    assert rel_l2(dq, dq_ref) <= GRAD_RELL2
    g = dlat.reshape(-1, cfg.d_l)[:cfg.R]
    assert rel_l2(g, dl_ref) <= GRAD_RELL2


def test_wait_limit_is_validated():
    L = lib()
    kp = torch.zeros(2, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    pool = L.lsr_page_pool_create(kp, kp.clone(), st)
    for bad in (-1, 4000001):
        with pytest.raises(L.LsrError):
            L.lsr_pool_set_wait_limit(pool, bad)
    L.lsr_pool_set_wait_limit(pool, 0)
