"""Host-side arithmetic of the split-key forward, checked on the CPU for the
decode shape (B1 Hq32 Hkv8, one query row, 131072 keys, d128) and others, at
every requested split count: the workspace the library asks for holds the
partial O and LSE arrays of the split count it will launch, that count never
exceeds the key tiles, and every split gets at least one key tile.  These are
the index ranges the split forward writes and the merge reads."""

import pytest

import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import build as libbuild


def _layout(rows, d, splits):
    o_bytes = (splits * rows * d * 4 + 255) // 256 * 256
    return o_bytes + (splits * rows * 4 + 255) // 256 * 256


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkg.load_library()


@pytest.mark.parametrize("shape", [(1, 32, 8, 1, 131072, 128), (1, 32, 8, 4, 131072, 128),
                                   (2, 4, 2, 3, 1000, 64), (1, 2, 1, 300, 4096, 128)])
def test_split_workspace_matches_launched_splits(lib, shape):
    B, Hq, Hkv, Nq, Nk, d = shape
    rows = B * Hq * Nq
    ktiles = -(-Nk // 128)
    for want in list(range(0, 257)):
        size = pkg.attn_fwd_split_workspace_size(B, Hq, Hkv, Nq, Nk, d, want)
        if want == 1 or (want > 0 and ktiles == 1):
            assert size == 0
            continue
        # The split count the library launches is the one whose layout has this size.
        cands = [s for s in range(1, ktiles + 1) if _layout(rows, d, s) == size]
        if size == 0:
            continue  # automatic choice of one split
        assert len(cands) == 1, (want, size)
        s = cands[0]
        assert 2 <= s <= min(ktiles, max(want, 1) if want else 64)
        per = -(-ktiles // s)
        # Every split [i*per, min((i+1)*per, ktiles)) holds at least one tile.
        assert all(i * per < ktiles for i in range(s)), (want, s, per)
        # The last split ends at the last tile: no key past Nk is addressed.
        assert (s - 1) * per < ktiles <= s * per
