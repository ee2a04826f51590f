"""Host logic of the CUDA-core decode kernel's work split (decode_gemv.cu,
split_rows), restated here: h block b -- the m * I / 32 routed ones, then the
shared expert's I / 32 -- goes to CTA b mod G, and each CTA gets a contiguous
range of output rows sized so that every CTA streams about the same bytes.
The ranges must tile [0, H) in CTA order for every kept count (every output
row is written exactly once), have lengths that are multiples of 4 (a down
stage's 4-row runs each belong to one expert), and the byte balance is what
makes the kernel's time the stream time.  The library's own computation
(moe_test_decode_split, host code) is checked against the restatement."""
import pytest

import block_quantized_expert_gb300 as bqe


def split_rows(G, m, H, I, nv=False, sh=False):
    sb = 16 if nv else 32
    FB = I // 32
    NBr = m * FB
    NB = NBr + (FB if sh else 0)
    Wr = 64 * (H // 2 + H // sb)
    Ws = 64 * H
    Wdn = m * (I // 2 + I // sb) + (I if sh else 0)
    Wg = (NBr * Wr + (NB - NBr) * Ws + H * Wdn) // G

    def cap(x):
        nr = (NBr - 1 - x) // G + 1 if x < NBr else 0
        nt = (NB - 1 - x) // G + 1 if x < NB else 0
        gu = nr * Wr + (nt - nr) * Ws
        return max(0, Wg - gu)

    total = sum(cap(x) for x in range(G))
    cut, pre = [], 0
    for x in range(G):
        r = x * H // G if total <= 0 else H * pre // total
        cut.append(min(H, (r + 2) // 4 * 4))
        pre += cap(x)
    cut.append(H)
    return cut


def stream_bytes(G, m, H, I, nv, sh, x, cut):
    sb = 16 if nv else 32
    FB = I // 32
    NBr, NB = m * FB, m * FB + (FB if sh else 0)
    nr = (NBr - 1 - x) // G + 1 if x < NBr else 0
    nt = (NB - 1 - x) // G + 1 if x < NB else 0
    gu = nr * 64 * (H // 2 + H // sb) + (nt - nr) * 64 * H
    rows = cut[x + 1] - cut[x]
    return gu, rows * (m * (I // 2 + I // sb) + (I if sh else 0))


SHAPES = [(4096, 2048), (2048, 1024), (8192, 2048), (8192, 1024), (2048, 2048)]
VARIANTS = [(False, False), (True, False), (False, True), (True, True)]


@pytest.mark.parametrize("H,I", SHAPES)
@pytest.mark.parametrize("G", [152, 148, 132, 160, 1, 7])
@pytest.mark.parametrize("nv,sh", VARIANTS)
def test_ranges_tile_the_rows(H, I, G, nv, sh):
    for m in range(1, 9):
        cut = split_rows(G, m, H, I, nv, sh)
        assert cut[0] == 0 and cut[-1] == H
        for x in range(G):
            assert cut[x + 1] >= cut[x]
            assert (cut[x + 1] - cut[x]) % 4 == 0


@pytest.mark.parametrize("G", [152, 148])
@pytest.mark.parametrize("nv,sh", VARIANTS)
def test_stream_bytes_balanced(G, nv, sh):
    """Decode shape, every kept count: no CTA streams more than the mean plus
    five down rows (the floor of the proportional cut and the rounding of
    both ends to multiples of 4), unless its gate/up blocks alone exceed the
    mean (few kept experts: those CTAs get no rows)."""
    H, I = 4096, 2048
    sb = 16 if nv else 32
    for m in range(1, 9):
        cut = split_rows(G, m, H, I, nv, sh)
        row = m * (I // 2 + I // sb) + (I if sh else 0)
        total = sum(sum(stream_bytes(G, m, H, I, nv, sh, x, cut)) for x in range(G))
        mean = total / G
        for x in range(G):
            gu, dn = stream_bytes(G, m, H, I, nv, sh, x, cut)
            if gu <= mean:
                assert gu + dn <= mean + 5 * row, (m, x, gu + dn, mean)
            else:
                assert dn == 0


def test_largest_range_bound():
    """The largest down range over kept counts 1..8 stays near 3H/G (the
    kernel sizes its shared partials with it)."""
    H, I, G = 4096, 2048, 152
    dmax = max(c[x + 1] - c[x] for m in range(1, 9) for c in [split_rows(G, m, H, I)] for x in range(G))
    assert dmax <= 3 * H // G + 6


@pytest.mark.parametrize("H,I", SHAPES)
@pytest.mark.parametrize("G", [152, 148, 7])
@pytest.mark.parametrize("nv,sh", VARIANTS)
def test_library_split_matches(H, I, G, nv, sh):
    for m in range(1, 9):
        assert bqe.moe_test_decode_split(G, m, H, I, nv, sh) == split_rows(G, m, H, I, nv, sh)


def test_library_split_rejects_bad_arguments():
    for args in [(0, 1, 4096, 2048), (152, 0, 4096, 2048), (152, 6, 4000, 2048), (152, 6, 4096, 16384)]:
        with pytest.raises(bqe.MoeError) as ei:
            bqe.moe_test_decode_split(*args)
        assert ei.value.status == bqe.MOE_ERR_INVALID_ARG
