"""How much Philox work exact pruning can skip on the headline recipe (bf16
logits, V = 151936, N(0, 4^2) plus the Zipf bumps, T = 1), in the oracle's
arithmetic ("Softmax-free GPU sampling", Background: score = x / T + g).

A 4-element group shares one Philox block, and no Gumbel value exceeds
G_MAX = g(1 - 2^-24), so a group may hold the row's winner only if its largest
logit reaches L - G_MAX (times T), L being any exact score of the row. These
tests measure that share at the row's final best score (the least Philox work
any exact method with this cap can do) and at the bound from the exact scores
of each 64-element block's largest logit, and check that the share is large
for this input: about half of the blocks are needed whatever the kernel does.
"""
import numpy as np

import oracle
import workloads as W

G_MAX = oracle.gumbel(1.0 - 2.0 ** -24)


def _row_scores(x: np.ndarray, seed: int, row: int, offset: int, T: float) -> np.ndarray:
    words = oracle.stream_words(seed, row, offset, 0, x.size)
    return x / T + oracle.gumbel_of_words(words)


def test_gumbel_cap_is_the_largest_value_of_the_uniform():
    assert abs(G_MAX - 16.6355) < 1e-3
    # every word's Gumbel value stays under the cap
    words = np.array([0, 1, 511, 512, 0xFFFFFDFF, 0xFFFFFE00, 0xFFFFFFFF], dtype=np.uint32)
    assert (oracle.gumbel_of_words(words) <= G_MAX).all()
    assert oracle.gumbel_of_words(np.array([0xFFFFFFFF], np.uint32))[0] == G_MAX


def test_share_of_groups_that_need_philox_on_the_headline_recipe():
    b = W.throughput(8)
    x = W.bf16_bits_to_f32(b.logits).astype(np.float64)
    T = 1.0
    final, blocks = [], []
    for r in range(b.B):
        s = _row_scores(x[r], int(b.seed[r]), r, int(b.offset[r]), T)
        L = s.max()
        xm = x[r].reshape(-1, 4).max(axis=1)
        final.append(float((xm >= (L - G_MAX) * T).mean()))
        # the bound from each 64-element block's largest logit, scored exactly
        blk = x[r].reshape(-1, 64)
        cand = blk.argmax(axis=1) + np.arange(blk.shape[0]) * 64
        Lb = s[cand].max()
        assert Lb <= L
        blocks.append(float((xm >= (Lb - G_MAX) * T).mean()))
    final, blocks = np.array(final), np.array(blocks)
    print("share of groups needing Philox: final bound %s (mean %.3f); "
          "64-element block maxima %s (mean %.3f)" % (np.round(final, 3), final.mean(),
                                                       np.round(blocks, 3), blocks.mean()))
    # about half of the blocks are needed at the best bound any exact method has
    assert 0.3 < final.mean() < 0.75
    assert (final > 0.2).all()
    # scoring every block maximum already gets (almost) there
    assert (blocks >= final).all()
    assert blocks.mean() - final.mean() < 0.05


def test_low_temperature_needs_little_philox():
    # the same recipe at T = 0.3: the cap shrinks relative to the logits' spread
    b = W.throughput(4)
    x = W.bf16_bits_to_f32(b.logits).astype(np.float64)
    T = 0.3
    for r in range(b.B):
        s = _row_scores(x[r], int(b.seed[r]), r, int(b.offset[r]), T)
        xm = x[r].reshape(-1, 4).max(axis=1)
        assert (xm >= (s.max() - G_MAX) * T).mean() < 0.1
