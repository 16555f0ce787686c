"""The jagged tile scheduler's rule in plain Python (test infrastructure).

Every (sequence b, head h, tile t) is one item whose cost is the number of inner steps
the kernel runs for it.  Sequences are ordered by total cost, heaviest first (cost
bucketed into 128 levels relative to the heaviest sequence, ties by b); the tiles of a
sequence are contiguous, heaviest first; the H heads of a tile are adjacent.  The GPU
tests compare the device-built lists with this; the CPU tests pin it on hand-worked
cases.
"""


BUCKETS = 128


def expected(lq, lk, H, tile, step, causal, key_major):
    """Sequences by total cost (bucketed relative to the heaviest), heaviest first, ties
    by index; a sequence's tiles contiguous, heaviest first; heads of a tile adjacent."""
    def cost(b, t):
        if not key_major:
            keys = min(lk[b], (t + 1) * tile) if causal else lk[b]
            return -(-keys // step)
        if not causal:
            return -(-lq[b] // step)
        return max(0, -(-lq[b] // step) - (t * tile) // step)

    ntile = [-(-(lk[b] if key_major else lq[b]) // tile) for b in range(len(lq))]
    total = [sum(cost(b, t) for t in range(ntile[b])) for b in range(len(lq))]
    top = max(total) if total else 0
    bucket = [total[b] * (BUCKETS - 1) // top if top > 0 else 0 for b in range(len(lq))]
    order = sorted(range(len(lq)), key=lambda b: (-bucket[b], b))
    out = []
    for b in order:
        n = ntile[b]
        for k in range(n):
            t = n - 1 - k if (causal and not key_major) else k
            for h in range(H):
                out.append((b, h, t, cost(b, t)))
    return out
