"""The LayerNorm launch choices, restated on the host, against the tolerance's bound on
the row sums' longest chain of additions (H // 128 + 32) and the ring's shared memory.

The single-CTA kernel takes batches of R rows (a power of two up to 32 filling two ring
slots of 64 KB, or one row a slot in a ring of 4H bytes), max(1, 8 / R) warps a row; a warp's
lane sums its half-vectors of 8 in four chains of two elements each, folds them (2),
the lanes (5) and the row's warps (8 / R - 1); up to 1024 columns 8 lanes take a row (the
lanes' butterfly: 3).  The cluster kernel does the same on a
column slice of hs = ceil(H / 8C) half-vectors (C = ceil(H / 4096)), R filling two ring
slots of 96 KB, then adds the C partial sums in rank order (C - 1).
"""
import oracle

RING = 64 * 1024
CLUSTER_RING = 96 * 1024


def pow2_batch(b, top=8):
    r = 1
    while r * 2 <= min(b, top):
        r *= 2
    return r


def single_cta_chain(H):
    nh = H // 8
    ring = max(RING, 2 * 2 * H)
    R = pow2_batch(ring // (2 * 2 * H), 32)
    if nh <= 128:  # up to 1024 columns: 8 lanes a row (butterfly of 3 steps), no warp totals
        assert R >= 16
        return 2 * -(-nh // 8) + 2 + 3, 2 * R * 2 * H
    wpr = max(1, 8 // R)
    return 2 * -(-nh // (32 * wpr)) + 2 + 5 + (wpr - 1), 2 * R * 2 * H


def cluster_chain(H):
    nh = H // 8
    C = -(-nh // 512)
    hs = -(-nh // C)
    last = nh - (C - 1) * hs
    R = pow2_batch(CLUSTER_RING // (2 * 16 * hs))
    wpr = 8 // R
    return 2 * -(-hs // (32 * wpr)) + 2 + 5 + (wpr - 1) + (C - 1), 2 * R * 16 * hs, C, last


def test_chain_and_ring_within_bounds_for_every_row_length():
    for H in range(16, 32768 + 1, 16):
        D, smem = single_cta_chain(H)
        assert D <= oracle.layernorm_chain_bound(H), H
        assert smem <= 128 * 1024, H
        if H > 4096:
            D, smem, C, last = cluster_chain(H)
            assert 2 <= C <= 8 and last > 0, H                # every slice has a CTA and columns
            assert D <= oracle.layernorm_chain_bound(H), H
            assert smem <= CLUSTER_RING, H
