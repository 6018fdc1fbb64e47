"""CPU pin of the block-summary definition the GPU tests compare attn_mask_blocks with:
the vectorised reshape-and-any against a loop over blocks and tiles written out, on
ragged sizes (a partial last block of rows, a partial last key tile, two words per
block) and with whole blocks and single tiles hidden."""
import numpy as np
import pytest

import synth
from tests.test_mask_blocks_gpu import summary_definition


def summary_loops(mask: np.ndarray) -> np.ndarray:
    m = np.asarray(mask, dtype=bool)
    lead = m.shape[:-2]
    nq, nk = m.shape[-2:]
    nblk, ntiles = -(-nq // 256), -(-nk // 128)
    wpb = -(-ntiles // 32)
    out = []
    for idx in np.ndindex(*lead):
        for p in range(nblk):
            words = [0] * wpb
            for j in range(ntiles):
                if m[idx][256 * p:256 * (p + 1), 128 * j:128 * (j + 1)].any():
                    words[j // 32] |= 1 << (j % 32)
            out.extend(words)
    return np.array(out, dtype=np.uint32)


@pytest.mark.parametrize("shape", [(1, 1), (300, 300), (2, 513, 4200), (2, 3, 256, 128), (700, 4097)])
def test_summary_definition_matches_loops(shape):
    m = synth.mask_random(500 + sum(shape), shape, 0.0005)
    if shape[-2] > 256:
        m[..., 256:512, :] = False  # a whole block hidden
    if shape[-1] > 128 * 32:
        m[..., :, 128 * 32:] = False
        m[..., 3, min(128 * 32 + 5, shape[-1] - 1)] = True  # one key in the first tile of word 1
    got = summary_definition(m)
    assert np.array_equal(got, summary_loops(m))


def test_summary_definition_worked_case():
    """A 300 x 300 mask with one visible key at (q = 260, k = 130): block 1 marks tile 1
    only, block 0 marks nothing."""
    m = np.zeros((300, 300), dtype=bool)
    m[260, 130] = True
    assert summary_definition(m).tolist() == [0, 0b10]
