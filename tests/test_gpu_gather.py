"""GPU parity of ds_chunk_topk_gather, through the C ABI.

The chosen chunk ids must equal the oracle's selection rule applied to the
same scores, bit for bit; the compact K/V bytes, positions and lengths must
equal the oracle's gather.  At full size the selection is also compared with
the selection made from float64 oracle scores: any difference must be a
near-tie (|s_k - s_(k+1)| <= 1e-3 s_k), and every planted salient chunk must
be chosen.
"""
import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
from oracle import ref
import helpers as H

pytestmark = pytest.mark.gpu


def _check_gather(wl, st, inp, step, scores_np, layout):
    H.check_gather(wl, st, inp, step, scores_np, layout)


def _set_scores(step, scores_np):
    step.scores.copy_(torch.from_numpy(scores_np.astype(np.float32)))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_select_and_gather_with_ties(layout, seed):
    wl = synth.tiny_workload(batch=4, chunk_size=32, top_k=5, window=70,
                             head_dim=128, num_q_heads=8, num_kv_heads=4)
    st, inp, mode = H.build_case(wl, layout=layout, seed=seed,
                                 ctx_lens=(2000, 500, 40, 0), tree_sizes=(3, 2, 2, 1))
    step = H.make_step(wl, inp, mode, layout)
    rng = np.random.default_rng(seed)
    scores = (rng.integers(0, 6, size=step.scores.shape) * 0.5).astype(np.float32)
    _set_scores(step, scores)
    step.gather()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    _check_gather(wl, st, inp, step, scores.astype(np.float64), layout)


def test_topk_larger_than_candidates_and_zero_k():
    wl = synth.tiny_workload(batch=2, chunk_size=16, top_k=50, window=16)
    st, inp, mode = H.build_case(wl, ctx_lens=(300, 33), tree_sizes=(2, 2), seed=4)
    step = H.make_step(wl, inp, mode)
    scores = np.random.default_rng(3).random(step.scores.shape).astype(np.float32)
    _set_scores(step, scores)
    step.gather()
    torch.cuda.synchronize()
    _check_gather(wl, st, inp, step, scores.astype(np.float64), "NHD")
    wl0 = wl.replace(top_k=0)
    step0 = H.make_step(wl0, inp, mode)
    _set_scores(step0, scores)
    step0.gather()
    torch.cuda.synchronize()
    _check_gather(wl0, st, inp, step0, scores.astype(np.float64), "NHD")


def test_many_candidates_radix_select():
    """Thousands of candidates with heavy ties exercise every radix digit."""
    wl = synth.tiny_workload(batch=2, chunk_size=16, top_k=700, window=100,
                             page_size=16)
    st, inp, mode = H.build_case(wl, ctx_lens=(60000, 9000), tree_sizes=(2, 2),
                                 seed=8)
    step = H.make_step(wl, inp, mode)
    rng = np.random.default_rng(2)
    s = rng.random(step.scores.shape).astype(np.float32)
    s[:, ::7] = 0.25                      # a large tie block
    s[0, 100:110] = np.float32(1e-30)     # tiny positives
    _set_scores(step, s)
    step.gather()
    torch.cuda.synchronize()
    _check_gather(wl, st, inp, step, s.astype(np.float64), "NHD")


@pytest.mark.parametrize("name", ["llama8b-32k", "llama8b-64k"])
def test_full_size_from_verify_scores(name):
    wl = synth.WORKLOADS[name]
    st, inp, mode = H.build_case(wl, layers=1)
    step = H.make_step(wl, inp, mode)
    step.verify_layer(0)
    step.gather()
    torch.cuda.synchronize()
    gs = step.scores.double().cpu().numpy()
    _check_gather(wl, st, inp, step, gs, "NHD")
    _, rs, _ = H.oracle_layer(wl, st, inp, 0, "NHD", step.max_chunks)
    H.check_selection_vs_f64(wl, st, gs, rs)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_gather_with_local_rope(layout, head_dim):
    """rope_base > 0: K rotated to its local position in the compact cache
    (vllm-diffspec README, "Architecture", dual-view draft cache).  Selection,
    positions, lengths and V stay byte-exact.  K against the oracle's
    once-rounded float64 rotation: the kernel reduces the angle exactly in
    64-bit fixed point, rounds it to float32 (at most 2^-24 pi off) and
    rotates in float32, an absolute error of at most ~1e-6 of the pair's
    norm before rounding, so |gpu - ref| <= ulp_bf16(ref) + 1e-6 * |pair|;
    and nearly every value is equal."""
    wl = synth.tiny_workload(batch=3, chunk_size=32, top_k=6, window=200,
                             head_dim=head_dim, num_q_heads=8, num_kv_heads=4)
    st, inp, mode = H.build_case(wl, layout=layout, seed=9,
                                 ctx_lens=(3000, 900, 100), tree_sizes=(3, 2, 2))
    step = H.make_step(wl, inp, mode, layout)
    rng = np.random.default_rng(3)
    scores = rng.random(step.scores.shape).astype(np.float32)
    _set_scores(step, scores)
    base = 500000.0
    ga = B.gather_args(step.scores, inp.ctx_lens, inp.src_k, inp.src_v, inp.page_table,
                       chunk_size=wl.chunk_size, top_k=wl.top_k, window=wl.window,
                       out_k=step.out_k, out_v=step.out_v,
                       out_positions=step.out_positions, out_len=step.out_len,
                       out_chunk_ids=step.out_chunk_ids, workspace=step.ws_gather,
                       kv_layout=layout, rope_base=base)
    B.ds_chunk_topk_gather(ga)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    exp = ref.gather_compact(H.bits(inp.src_k), H.bits(inp.src_v), st.page_table.numpy(),
                             st.ctx_lens, scores.astype(np.float64), wl.page_size,
                             wl.chunk_size, wl.top_k, wl.window, step.capacity,
                             layout=layout, rope_base=base)
    np.testing.assert_array_equal(step.out_len.cpu().numpy(), exp["out_len"])
    np.testing.assert_array_equal(step.out_positions.cpu().numpy(), exp["positions"])
    ok, ov = H.bits(step.out_k), H.bits(step.out_v)
    exact = total = 0
    for b in range(wl.batch):
        n = exp["out_len"][b]
        np.testing.assert_array_equal(ov[b, :n], exp["out_v"][b, :n])
        g = ref.bf16_bits_to_f64(ok[b, :n])
        o = ref.bf16_bits_to_f64(exp["out_k"][b, :n])
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o), 1e-30))) - 7)
        half = head_dim // 2
        pair = np.sqrt(o[..., :half] ** 2 + o[..., half:] ** 2)
        pair = np.concatenate([pair, pair], axis=-1)
        tol = ulp + 1e-6 * pair
        assert (np.abs(g - o) <= tol).all(), f"seq {b}: max err {np.abs(g - o).max()}"
        exact += int((ok[b, :n] == exp["out_k"][b, :n]).sum())
        total += ok[b, :n].size
    assert exact >= 0.995 * total, (exact, total)


@pytest.mark.parametrize("rope", [0.0, 500000.0])
def test_compact_append_between_retrievals(rope):
    """ds_compact_append after a GPU gather: the tokens committed since are
    appended behind the last row (vllm-diffspec README, "What DiffSpec Does"
    item 4); compared with the oracle's append of the oracle's gather.  A
    sequence whose rows would not fit is flagged and left as it was."""
    wl = synth.tiny_workload(batch=3, chunk_size=32, top_k=3, window=100,
                             head_dim=128, num_q_heads=8, num_kv_heads=4)
    # the source pages must cover the appended tokens: contexts as they
    # will be after the append, retrieval made at the earlier lengths
    old = [900, 300, 1000]
    new = [917, 300, 1400]                      # seq 2 overflows the capacity
    st, inp, mode = H.build_case(wl, layout="NHD", seed=21, ctx_lens=new,
                                 tree_sizes=(2, 2, 2))
    step = H.make_step(wl, inp, mode, "NHD")
    rng = np.random.default_rng(5)
    scores = rng.random(step.scores.shape).astype(np.float32)
    _set_scores(step, scores)
    dev = step.out_k.device
    i32 = dict(dtype=torch.int32, device=dev)
    old_t = torch.tensor(old, **i32)
    cap = step.capacity + 64                    # room for appended rows
    out_k = torch.zeros(3, cap, 4, 128, dtype=torch.bfloat16, device=dev)
    out_v = torch.zeros_like(out_k)
    pos = torch.empty(3, cap, **i32)
    olen = torch.empty(3, **i32)
    ids = torch.empty(3, wl.top_k, **i32)
    ga = B.gather_args(step.scores, old_t, inp.src_k, inp.src_v, inp.page_table,
                       chunk_size=wl.chunk_size, top_k=wl.top_k, window=wl.window,
                       out_k=out_k, out_v=out_v, out_positions=pos, out_len=olen,
                       out_chunk_ids=ids, workspace=step.ws_gather, rope_base=rope)
    B.ds_chunk_topk_gather(ga)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    aa = B.append_args(inp.src_k, inp.src_v, inp.page_table, old_t,
                       torch.tensor(new, **i32), out_k=out_k, out_v=out_v,
                       out_positions=pos, out_len=olen, workspace=ws, rope_base=rope)
    B.ds_compact_append(aa)
    torch.cuda.synchronize()
    assert B.ds_device_status(ws) & B.DS_DEV_BAD_LENGTH          # sequence 2
    kb, vb = H.bits(inp.src_k), H.bits(inp.src_v)
    first = ref.gather_compact(kb, vb, st.page_table.numpy(), old, scores.astype(np.float64),
                               wl.page_size, wl.chunk_size, wl.top_k, wl.window,
                               cap, rope_base=rope)
    exp = ref.compact_append(first, kb, vb, st.page_table.numpy(), old, new,
                             wl.page_size, rope_base=rope)
    assert olen.cpu().numpy().tolist() == exp["out_len"].tolist()
    assert exp["out_len"].tolist() == [first["out_len"][0] + 17, first["out_len"][1],
                                       first["out_len"][2]]
    np.testing.assert_array_equal(pos.cpu().numpy(), exp["positions"])
    ok, ov = H.bits(out_k), H.bits(out_v)
    for b in range(3):
        n = exp["out_len"][b]
        np.testing.assert_array_equal(ov[b, :n], exp["out_v"][b, :n])
        if rope == 0.0:
            np.testing.assert_array_equal(ok[b, :n], exp["out_k"][b, :n])
        else:
            g = ref.bf16_bits_to_f64(ok[b, :n])
            o = ref.bf16_bits_to_f64(exp["out_k"][b, :n])
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o), 1e-30))) - 7)
            pair = np.sqrt(o[..., :64] ** 2 + o[..., 64:] ** 2)
            pair = np.concatenate([pair, pair], axis=-1)
            assert (np.abs(g - o) <= ulp + 1e-6 * pair).all()
