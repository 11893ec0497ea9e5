"""Device-resident bad values are caught by the kernels' own bounds checks:
no out-of-bounds access, a sticky status bit in the workspace, and the
valid sequences of the batch still match the oracle."""
import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
import helpers as H

pytestmark = pytest.mark.gpu


def _case(**kw):
    wl = synth.tiny_workload(batch=2, **kw)
    st, inp, mode = H.build_case(wl, ctx_lens=(200, 300), tree_sizes=(5, 6),
                                 seed=31, mode="reject")
    return wl, st, inp


def test_bad_page_id_sets_flag_and_spares_other_sequence():
    wl, st, inp = _case()
    step = H.make_step(wl, inp, "reject", out_dtype=torch.float32)
    inp.page_table[0, 3] = st.num_pages + 7        # out of the pool
    step.verify_layer(0)
    step.gather()
    torch.cuda.synchronize()
    assert B.ds_device_status(step.ws_verify) & B.DS_DEV_BAD_PAGE
    assert B.ds_device_status(step.ws_gather) & B.DS_DEV_BAD_PAGE
    # the host table st.page_table still holds the valid ids
    o, _, _ = H.oracle_layer(wl, st, inp, 0, "NHD", step.max_chunks)
    n1 = st.tree_offsets[1]
    H.assert_attention_close(step.out[0][n1:], o[n1:], "seq 1")
    B.ds_workspace_init(step.ws_verify)
    assert B.ds_device_status(step.ws_verify) == 0


def test_bad_parent_and_bad_length_flags():
    wl, st, inp = _case()
    step = H.make_step(wl, inp, "reject")
    inp.parents[st.tree_offsets[1] + 2] = 4        # not an earlier node
    step.verify_layer(0)
    torch.cuda.synchronize()
    assert B.ds_device_status(step.ws_verify) & B.DS_DEV_BAD_TREE
    B.ds_workspace_init(step.ws_verify)
    inp.ctx_lens[0] = 10 ** 7                      # beyond the page table
    step.verify_layer(0)
    torch.cuda.synchronize()
    assert B.ds_device_status(step.ws_verify) & B.DS_DEV_BAD_LENGTH


def test_bad_token_flag():
    wl, st, inp = _case()
    step = H.make_step(wl, inp, "reject")
    inp.draft_tokens[1] = wl.vocab + 3
    step.accept()
    torch.cuda.synchronize()
    assert B.ds_device_status(step.ws_accept) & B.DS_DEV_BAD_TOKEN


def test_bad_tree_offsets_flag_in_accept():
    """An offset past the node arrays: the walk flags the sequence and gives
    it n = 0, bonus -1; the node pass gives it no children, so no parent or
    token read leaves the arrays."""
    wl, st, inp = _case()
    step = H.make_step(wl, inp, "reject")
    inp.tree_offsets[2] = st.n_nodes + 5
    step.accept()
    torch.cuda.synchronize()
    assert B.ds_device_status(step.ws_accept) & B.DS_DEV_BAD_TREE
    assert int(step.out_n[1]) == 0 and int(step.out_bonus[1]) == -1
