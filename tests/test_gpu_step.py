"""The end-to-end step from pinned host inputs (VerifyStep.run_from_host:
copies on a side stream, each layer's verify waiting only for its own Q)
gives bit-identical results to the step on device-resident inputs, and so
does the same step captured once as a CUDA graph and replayed."""
import pytest
import torch

from long_context_speculative_ds_gb300 import synth
import helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["greedy", "reject"])
def test_run_from_host_matches_resident(mode):
    wl = synth.tiny_workload(batch=3, vocab=500, max_depth=6, max_branch=3)
    st, inp, _ = H.build_case(wl, mode=mode, seed=21, layers=3,
                              ctx_lens=[300, 77, 1000], tree_sizes=[12, 1, 40])
    step = H.make_step(wl, inp, mode)
    step.run()
    torch.cuda.synchronize()
    names = ("out_path", "out_n", "out_bonus", "out_chunk_ids", "out_len",
             "out_k", "out_v", "out_positions", "scores")
    want = {n: getattr(step, n).clone() for n in names}
    want_o = [o.clone() for o in step.out]
    n_len = want["out_len"].cpu()

    pin = lambda t: None if t is None else t.cpu().pin_memory()
    host = type(inp)(
        page_table=pin(inp.page_table), ctx_lens=pin(inp.ctx_lens),
        tree_offsets=pin(inp.tree_offsets), parents=pin(inp.parents),
        q=[pin(x) for x in inp.q], k_cache=[], v_cache=[], src_k=None, src_v=None,
        target_logits=pin(inp.target_logits), draft_logits=pin(inp.draft_logits),
        draft_tokens=pin(inp.draft_tokens), uniforms=pin(inp.uniforms))
    # clobber every per-step device input and every output
    for t in [inp.target_logits, inp.draft_tokens] + list(inp.q):
        t.zero_()
    if inp.draft_logits is not None:
        inp.draft_logits.zero_()
    if inp.uniforms is not None:
        inp.uniforms.fill_(0.5)
    for n in names:
        getattr(step, n).zero_()
    for o in step.out:
        o.zero_()
    host_out = {n: torch.empty_like(getattr(step, n), device="cpu").pin_memory()
                for n in ("out_path", "out_n", "out_bonus", "out_chunk_ids", "out_len")}
    h2d, d2h = step.run_from_host(host, host_out)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    assert h2d > 0 and d2h > 0
    for n in names:
        a, b = getattr(step, n), want[n]
        if n in ("out_k", "out_v", "out_positions"):
            for bi in range(wl.batch):     # rows past out_len are not written
                k = int(n_len[bi])
                assert torch.equal(a[bi, :k], b[bi, :k]), n
        else:
            assert torch.equal(a, b), n
    for l, (a, b) in enumerate(zip(step.out, want_o)):
        assert torch.equal(a, b), f"layer {l} attention"
    for n in host_out:
        assert torch.equal(host_out[n], want[n].cpu()), n


@pytest.mark.parametrize("mode", ["greedy", "reject"])
def test_captured_step_replays_the_eager_step(mode):
    """capture_from_host + replay: the same results as the eager
    run_from_host, and a replay reads the pinned host inputs as they are
    when it runs (new draft tokens change the accepted paths the same way
    in both)."""
    wl = synth.tiny_workload(batch=3, vocab=500, max_depth=6, max_branch=3)
    st, inp, _ = H.build_case(wl, mode=mode, seed=33, layers=2,
                              ctx_lens=[300, 77, 1000], tree_sizes=[12, 1, 40])
    step = H.make_step(wl, inp, mode)
    pin = lambda t: None if t is None else t.cpu().pin_memory()
    host = type(inp)(
        page_table=pin(inp.page_table), ctx_lens=pin(inp.ctx_lens),
        tree_offsets=pin(inp.tree_offsets), parents=pin(inp.parents),
        q=[pin(x) for x in inp.q], k_cache=[], v_cache=[], src_k=None, src_v=None,
        target_logits=pin(inp.target_logits), draft_logits=pin(inp.draft_logits),
        draft_tokens=pin(inp.draft_tokens), uniforms=pin(inp.uniforms))
    small = ("out_path", "out_n", "out_bonus", "out_chunk_ids", "out_len")
    host_out = {n: torch.empty_like(getattr(step, n), device="cpu").pin_memory()
                for n in small}

    def snapshot():
        return {n: host_out[n].clone() for n in small}, [o.clone() for o in step.out]

    step.run_from_host(host, host_out)
    torch.cuda.synchronize()
    want, want_o = snapshot()
    bytes_eager = step.run_from_host(host, host_out)
    torch.cuda.synchronize()
    assert step.capture_from_host(host, host_out) == bytes_eager
    for n in small:
        host_out[n].zero_()
    for o in step.out:
        o.zero_()
    step.replay()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    got, got_o = snapshot()
    for n in small:
        assert torch.equal(got[n], want[n]), n
    for a, b in zip(got_o, want_o):
        assert torch.equal(a, b)

    # new drafted tokens in the pinned buffer: replay and eager agree
    g = torch.Generator().manual_seed(5)
    host.draft_tokens.copy_(torch.randint(0, wl.vocab, host.draft_tokens.shape,
                                          generator=g, dtype=torch.int32))
    step.replay()
    torch.cuda.synchronize()
    got2, _ = snapshot()
    step.run_from_host(host, host_out)
    torch.cuda.synchronize()
    want2, _ = snapshot()
    for n in small:
        assert torch.equal(got2[n], want2[n]), n
