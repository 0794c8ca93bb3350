"""The step from pinned host memory (Step.run_host): q_lat crosses on a second
stream while compression, scoring and selection run, and the attention waits
for it through kp_forward_args.q_lat_ready.  Every output must equal, bit for
bit, a run of the same step on a fresh session with the inputs already on the
device, eagerly and inside a captured CUDA graph, with and without a shared
selection and in both select modes."""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp

pytestmark = pytest.mark.gpu


def _reference(wl, mode, share):
    sess, step = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode))
    if share is not None:
        step.set_share(share)
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    return step, PL.gpu_pooled_of_seq(sess, wl, 0)


def _host_step(wl, mode, share):
    sess, step = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode))
    if share is not None:
        step.set_share(share)
    in_buf, out_buf = step.pack_io()
    h_in = torch.empty(in_buf.numel(), dtype=torch.uint8).pin_memory()
    h_in.copy_(in_buf)
    h_out = torch.empty(out_buf.numel(), dtype=torch.uint8).pin_memory()
    return sess, step, in_buf, out_buf, h_in, h_out


def _same(step, ref, h_out, out_buf, share=None):
    assert torch.equal(step.out, ref.out) and torch.equal(step.lse, ref.lse)
    g_idx, g_n = step.pool_idx.cpu().numpy(), step.n_sel.cpu().numpy()
    r_idx, r_n = ref.pool_idx.cpu().numpy(), ref.n_sel.cpu().numpy()
    for q in range(len(r_n)):
        if share is not None and share[q] >= 0:
            continue                # a shared query's row is not written
        assert g_n[q] == r_n[q]
        assert np.array_equal(g_idx[q, :r_n[q]], r_idx[q, :r_n[q]])
    assert np.array_equal(h_out.numpy(), out_buf.cpu().numpy())   # the host copy is the device result


@pytest.mark.parametrize("mode,share", [(kp.SELECT_STAGED, None), (kp.SELECT_FUSED, None),
                                        (kp.SELECT_AUTO, "mtp")])
def test_run_host_equals_run(mode, share):
    wl = KI.make(KI.Spec("hostio", [5000, 9003, 3001], [2, 2, 2], topk_tokens=512, seed=81))
    share = [-1, 0, -1, 2, -1, 4] if share == "mtp" else None
    ref, ref_pooled = _reference(wl, mode, share)
    sess, step, in_buf, out_buf, h_in, h_out = _host_step(wl, mode, share)
    in_buf.zero_()                  # every input must arrive through the copies
    step.out.zero_()
    step.run_host(h_in, h_out)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    _same(step, ref, h_out, out_buf, share)
    assert np.array_equal(PL.gpu_pooled_of_seq(sess, wl, 0), ref_pooled)


def test_run_host_in_a_cuda_graph():
    wl = KI.make(KI.Spec("hostio", [33000, 20001, 4099, 8192], [1, 1, 1, 1], topk_tokens=2048, seed=82))
    ref, _ = _reference(wl, kp.SELECT_AUTO, None)
    sess, step, in_buf, out_buf, h_in, h_out = _host_step(wl, kp.SELECT_AUTO, None)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step.run_host(h_in, h_out)          # eager first: the events and the copy stream exist
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step.run_host(h_in, h_out)
        for _ in range(2):
            in_buf.zero_()
            step.out.zero_()
            h_out.zero_()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert int(sess.status.item()) == 0
            _same(step, ref, h_out, out_buf)


def test_run_host_without_queries():
    from dsa_indexer_sparse_kpool_b300.session import Step, build_session
    wl = KI.make(KI.Spec("hostio", [1030, 515], [6, 3], topk_tokens=256, seed=83))
    sess = build_session(PL.cfg_of(wl), wl.lens.tolist(), wl.prev_len.tolist(), wl.tok_off.tolist(),
                         wl.pool_off.tolist(), wl.pool_rows, wl.latent, wl.keys, wl.gates, wl.ape)
    counts = [int(x) for x in (wl.lens - wl.prev_len)]
    idx = torch.cat([torch.arange(int(wl.tok_off[b] + wl.prev_len[b]), int(wl.tok_off[b] + wl.lens[b]))
                     for b in range(wl.B)])
    step = Step(sess, wl.prev_len.tolist(), counts, wl.keys[idx], wl.gates[idx], [], [], wl.q_idx[:0], wl.w[:0],
                wl.q_lat[:0])
    in_buf, out_buf = step.pack_io()
    h_in = torch.empty(in_buf.numel(), dtype=torch.uint8).pin_memory()
    h_in.copy_(in_buf)
    h_out = torch.empty(out_buf.numel(), dtype=torch.uint8).pin_memory()
    in_buf.zero_()
    step.run_host(h_in, h_out)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    PL.check_pooled(sess, wl)


def test_run_host_needs_pack_io_and_matching_buffers():
    wl = KI.make(KI.Spec("hostio", [3001], [2], topk_tokens=256, seed=84))
    _, step = PL.make_gpu(wl)
    with pytest.raises(RuntimeError):
        step.run_host(torch.empty(1, dtype=torch.uint8), torch.empty(1, dtype=torch.uint8))
    in_buf, out_buf = step.pack_io()
    with pytest.raises(ValueError):
        step.run_host(torch.empty(in_buf.numel() + 1, dtype=torch.uint8).pin_memory(),
                      torch.empty(out_buf.numel(), dtype=torch.uint8).pin_memory())


@pytest.mark.parametrize("chunk", [256, 128])
def test_run_host_chunked_pipeline_equals_run(chunk):
    # 600 queries of one sequence, as in a prefill chunk: two chunks of 300
    # queries, or four of 150, each with its own q_lat copy, attention and
    # copy back; eagerly, then replayed from a captured graph
    wl = KI.make(KI.Spec("hostio", [20000], [600], topk_tokens=2048, seed=85))
    ref, ref_pooled = _reference(wl, kp.SELECT_AUTO, None)
    sess, step, in_buf, out_buf, h_in, h_out = _host_step(wl, kp.SELECT_AUTO, None)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        in_buf.zero_()
        step.out.zero_()
        step.run_host(h_in, h_out, chunk_queries=chunk)
        torch.cuda.synchronize()
        assert int(sess.status.item()) == 0
        assert len(step._chunked["bounds"]) == 600 // chunk
        _same(step, ref, h_out, out_buf)
        assert np.array_equal(PL.gpu_pooled_of_seq(sess, wl, 0), ref_pooled)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step.run_host(h_in, h_out, chunk_queries=chunk)
        in_buf.zero_()
        step.out.zero_()
        h_out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(sess.status.item()) == 0
        _same(step, ref, h_out, out_buf)


def test_run_host_rejects_small_chunks():
    wl = KI.make(KI.Spec("hostio", [3001], [2], topk_tokens=256, seed=86))
    _, step = PL.make_gpu(wl)
    in_buf, out_buf = step.pack_io()
    h_in = torch.empty(in_buf.numel(), dtype=torch.uint8).pin_memory()
    h_out = torch.empty(out_buf.numel(), dtype=torch.uint8).pin_memory()
    with pytest.raises(ValueError):
        step.run_host(h_in, h_out, chunk_queries=64)


@pytest.mark.parametrize("mode,page_tokens", [(kp.SELECT_FUSED, None), (kp.SELECT_STAGED, 256)])
def test_run_host_chunked_fused_select_and_pages(mode, page_tokens):
    # the selection-only call through the fused score-and-select kernel, and
    # the chunked attention on paged caches, each against the device-only step
    wl = KI.make(KI.Spec("hostio", [20000], [600], topk_tokens=2048, seed=87))
    _, ref = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode), page_tokens=page_tokens)
    ref.run()
    torch.cuda.synchronize()
    sess, step = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode), page_tokens=page_tokens)
    in_buf, out_buf = step.pack_io()
    h_in = torch.empty(in_buf.numel(), dtype=torch.uint8).pin_memory()
    h_in.copy_(in_buf)
    h_out = torch.empty(out_buf.numel(), dtype=torch.uint8).pin_memory()
    in_buf.zero_()
    step.out.zero_()
    step.run_host(h_in, h_out, chunk_queries=256)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    assert len(step._chunked["bounds"]) == 2
    _same(step, ref, h_out, out_buf)
