"""Host logic of the CUDA-core decode kernel's work split (decode_gemv.cu,
cut_rows / down_rows), restated here: gate/up block b goes to CTA b mod G, and each CTA
gets a contiguous range of output rows sized so that every CTA streams about
the same bytes.  The ranges must tile [0, H) in CTA order for every kept
count (every output row is written exactly once), and the byte balance is
what makes the kernel's time the stream time."""
import pytest

SEG = 1024


def cut_rows(c, G, m, H, I):
    """Start row of CTA c: the rows cut in proportion to the CTAs' capacities
    for down bytes, rounded to a multiple of 4 (a down stage's 4-row runs
    then each belong to one expert)."""
    FB = I // 32
    NB = m * FB
    q0, rr = NB // G, NB % G
    Wgu = 64 * (H // 2 + H // 32)
    Wdn = m * (I // 2 + I // 32)
    Wg = (NB * Wgu + H * Wdn) // G
    capA = max(0, Wg - (q0 + 1) * Wgu)
    capB = max(0, Wg - q0 * Wgu)

    def cap(x):
        return min(x, rr) * capA + max(0, x - rr) * capB

    total = cap(G)
    r = c * H // G if total <= 0 else H * cap(c) // total
    return (r + 2) // 4 * 4


def down_rows(c, G, m, H, I):
    r0 = cut_rows(c, G, m, H, I)
    r1 = H if c + 1 == G else cut_rows(c + 1, G, m, H, I)
    r1 = min(r1, H)
    return min(r0, r1), r1


SHAPES = [(4096, 2048), (1024, 1024), (2048, 4096), (8192, 4096), (8192, 1024)]


@pytest.mark.parametrize("H,I", SHAPES)
@pytest.mark.parametrize("G", [152, 148, 132, 160, 1, 7])
def test_ranges_tile_the_rows(H, I, G):
    for m in range(1, 9):
        prev = 0
        for c in range(G):
            r0, r1 = down_rows(c, G, m, H, I)
            assert r0 == prev and r1 >= r0
            assert (r1 - r0) % 4 == 0
            prev = r1
        assert prev == H


@pytest.mark.parametrize("G", [152, 148])
def test_stream_bytes_balanced(G):
    """Decode shape, every kept count: no CTA streams more than the mean plus
    five down rows (the floor of the proportional cut and the rounding of
    both ends to multiples of 4), unless its gate/up blocks alone exceed the
    mean (few kept experts: those CTAs get no rows)."""
    H, I = 4096, 2048
    FB = I // 32
    Wgu = 64 * (H // 2 + H // 32)
    for m in range(1, 9):
        Wdn = m * (I // 2 + I // 32)
        NB = m * FB
        total = NB * Wgu + H * Wdn
        mean = total / G
        for c in range(G):
            nb = (NB - c + G - 1) // G if c < NB else 0
            r0, r1 = down_rows(c, G, m, H, I)
            b = nb * Wgu + (r1 - r0) * Wdn
            if nb * Wgu <= mean:
                assert b <= mean + 5 * Wdn, (m, c, b, mean)
            else:
                assert r1 == r0


def test_largest_range_bound():
    """The largest down range over kept counts 1..8 stays near 3H/G (the
    kernel sizes its shared partials with it)."""
    H, I, G = 4096, 2048, 152
    dmax = max(down_rows(c, G, m, H, I)[1] - down_rows(c, G, m, H, I)[0]
               for m in range(1, 9) for c in range(G))
    assert dmax <= 3 * H // G + 6
