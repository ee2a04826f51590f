"""The stream-K partition of the one-token decode kernel, checked on the CPU
for every shape the kernel accepts and several SM counts.

The partition is integer arithmetic (SegIter in gemm_tc.cu: a phase of
`tiles` x `KB` K-stages cut into G equal contiguous ranges, one per CTA);
this test restates it and checks the properties the kernel relies on:

- every K-stage of a phase belongs to exactly one CTA, and every CTA gets at
  least one when the phase is split (one K-stage per CTA is the decode
  minimum, so a token that keeps one expert still uses the whole grid);
- a cut tile is finished by the CTA holding its first K-stage, whose 32
  waiting lanes cover the later pieces: at most 32 of them;
- a CTA's later pieces are always its first segment (parking slot 0), and a
  CTA range holds at most two segments;
- a down-phase range spans at most two experts (the h rows of two experts
  fit the CTA's shared memory).
"""
import pytest

KMAX = 8  # the decode kernel's largest top-k


def seg_ranges(tiles, KB, G, min_stages):
    """Per CTA the list of (tile, kb0, kb1, first_cta, last_cta) segments."""
    total = tiles * KB
    split = tiles < 4 * G and total >= min_stages * G

    def owner(gs):
        return ((gs + 1) * G + total - 1) // total - 1

    out = []
    for c in range(G):
        segs = []
        if split:
            g, gend = c * total // G, (c + 1) * total // G
            while g < gend:
                t, kb0 = g // KB, g % KB
                kb1 = min(KB, kb0 + (gend - g))
                segs.append((t, kb0, kb1, owner(t * KB), owner(t * KB + KB - 1)))
                g += kb1 - kb0
        else:
            for t in range(c, tiles, G):
                segs.append((t, 0, KB, c, c))
        out.append(segs)
    return split, out


def decode_supported(H, I, k, G):
    return H % 256 == 0 and H <= 4096 and I <= 2048 and k <= KMAX and k * (H // 256) <= 2 * G


SHAPES = [(H, I) for H in (256, 1024, 2048, 4096) for I in (128, 512, 1024, 2048)]


@pytest.mark.parametrize("G", [120, 132, 148, 152, 160])
@pytest.mark.parametrize("H,I", SHAPES)
def test_decode_partition_properties(G, H, I):
    for k in range(1, KMAX + 1):
        if not decode_supported(H, I, k, G):
            continue
        for down in (False, True):
            MT = H // 256 if down else I // 128
            KB = I // 128 if down else H // 128
            tiles = k * MT
            split, per_cta = seg_ranges(tiles, KB, G, 1)
            seen, cut = {}, {}
            for c, segs in enumerate(per_cta):
                if split:
                    assert len(segs) <= 2
                for j, (t, kb0, kb1, first, last) in enumerate(segs):
                    for kb in range(kb0, kb1):
                        assert (t, kb) not in seen, (G, H, I, k, down, t, kb)
                        seen[(t, kb)] = c
                    if first != last:
                        cut[t] = (first, last)
                        assert last - first <= 32, (G, H, I, k, down, t, first, last)
                        if c != first:
                            assert j == 0  # a later piece is the CTA's first segment: slot 0
                        else:
                            assert j == len(segs) - 1  # the finishing piece is its last
                    else:
                        assert first == c
            assert len(seen) == tiles * KB
            for t, (first, last) in cut.items():
                # finished by the CTA holding the tile's first stage; the last holds its end
                assert seen[(t, 0)] == first and seen[(t, KB - 1)] == last
            if split:
                assert all(len(s) >= 1 for s in per_cta)
            if down:
                for segs in per_cta:
                    experts = sorted({t // MT for t, *_ in segs})
                    assert len(experts) <= 2, (G, H, I, k, experts)


def test_one_kept_expert_uses_the_whole_grid():
    # H 4096, I 2048, one expert: 512 gate/up and 256 down stages on 152 SMs
    for down, (tiles, KB) in ((False, (16, 32)), (True, (16, 16))):
        split, per_cta = seg_ranges(tiles, KB, 152, 1)
        assert split and all(per_cta)
        # the grouped kernels' minimum of four stages per CTA would not split
        assert not seg_ranges(tiles, KB, 152, 4)[0]
