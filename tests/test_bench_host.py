"""Host-side logic of bench.py that decides what the timed region measures:
how many resident input copies keep the calls from being served from L2, and
the order in which the captured graphs walk through them."""
import bench

L2 = 126 << 20


def walk(R, G, K):
    """Copies used by the timed region's K calls: graphs[t % NG] for the
    first K / G - 1 replays, then the event graph on the copies next in turn."""
    plan = bench.graph_copies(R, G)
    NG = len(plan)
    seq = []
    for t in range(K // G - 1):
        seq += plan[t % NG]
    seq += plan[(K // G - 1) % NG]
    return seq


def test_large_inputs_keep_two_alternating_copies():
    # the mixed serving batch: 1.24 GB of logits and draft probs per call
    R = bench.input_copies(1_240_000_000, L2, 10)
    assert R == 2
    assert bench.graph_copies(R, 10) == [[0, 1] * 5]


def test_small_inputs_rotate_past_twice_l2():
    for call_bytes in (512_000, 17_800_000, 76_000_000, 140_000_000):
        for G in (10, 5, 4):
            R = bench.input_copies(call_bytes, L2, G)
            assert R * call_bytes >= 2 * L2
            assert R == 2 or R % G == 0
            assert R * call_bytes < 2 * L2 + G * call_bytes + 2 * call_bytes  # no more than needed


def test_walk_never_reuses_a_copy_within_r_calls():
    for call_bytes, G, K in ((17_800_000, 10, 500), (512_000, 10, 2000), (76_000_000, 10, 500),
                             (1_240_000_000, 10, 2000), (1_240_000_000, 3, 9), (17_800_000, 4, 8)):
        R = bench.input_copies(call_bytes, L2, G)
        seq = walk(R, G, K)
        assert len(seq) == K
        assert seq == [c % R for c in range(K)] or (R == 2 and seq == [c % 2 for c in range(K)])
        for a in range(0, K - R + 1, max(1, R // 2)):
            assert len(set(seq[a:a + R])) == R
