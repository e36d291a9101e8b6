"""GPU parity at the full sizes of the four work lists, in the launch configuration
bench.py times (one persistent launch per stage over the whole list): every image row
of the image-only list; >= 4096 seeded random query rows per (item, head) plus tile
edges for the video shards; for the training step, every forward row, and dQ / dK / dV
on >= 4096 seeded query / KV rows of every head of every item (N(0,1) and structured
inputs)."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300.workloads import config_images, config_long_video, config_mixed, config_training
from tests.gpu_util import Run, all_heads, check_forward_pairs, check_gradients, oracle_pairs

pytestmark = pytest.mark.gpu


def test_images_full_all_rows():
    Run(config_images(), seed=0).check_forward()


def test_mixed_shards_full_sampled_rows():
    Run(config_mixed(), seed=0).check_forward(sample=4096)


def test_long_video_k8_full_sampled_rows():
    Run(config_long_video(), seed=0).check_forward(sample=4096)


@pytest.mark.parametrize("structured", [False, True], ids=["randn", "structured"])
def test_training_full(structured):
    """The benched training step at full size: forward O / LSE of every row, and dQ on
    >= 4096 seeded query rows and dK / dV on >= 4096 seeded KV rows (all rows where an
    item has fewer), against the oracle's gradient with the final (merged) O and LSE.
    N(0,1) inputs: every head of every item, plus the whole-item gradient sums.
    Structured inputs (Q x 4, V + 3): the first and last head of every item."""
    w = config_training()
    r = Run(w, seed=1 if structured else 0, structured=structured, backward=True)
    heads_of = ({i: sorted({it.h_lo, it.h_hi - 1}) for i, it in enumerate(r.items)} if structured
                else all_heads(r))
    own, final = oracle_pairs(r, heads_of)
    check_forward_pairs(r, own, final)
    check_gradients(r, final, q_sample=4096, kv_sample=4096, seed=40 if structured else 0)
    if structured:
        return
    for i, it in enumerate(r.items):
        # whole items, every head: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i
        if not it.emit_lse and it.nq == it.seq_len and it.nh == w.n_heads and it.nkv == it.seq_len:
            s = it.seq_offset
            dv, dk = r.grad(i, "dv"), r.grad(i, "dk")
            np.testing.assert_allclose(dv.sum(axis=0), r.do[s:s + it.seq_len].sum(axis=0), atol=5e-2)
            np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=5e-2)
