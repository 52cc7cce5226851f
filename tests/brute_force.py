"""Pure-Python brute force for the PLE n-gram row-id hash (a test pin).

It shares nothing with the C oracle: no packed window and no cummax scan.
For every token t and shift s it reads the id s places to the left straight
from the flat ids or the carried context, with the addressing rule of
FreeToken PR #338 ("perf(ple): fuse the n-gram row-id hash into one Triton
kernel", section "What", second observation), and decides validity by
walking the whole interval [p-s, p-1] (first observation) one cell at a time.
Arithmetic uses Python integers masked to 64 bits and Python's floored %.
"""

MASK = (1 << 64) - 1


def to_signed(x: int) -> int:
    x &= MASK
    return x - (1 << 64) if x >> 63 else x


def brute_row_ids(ids, req, local, ctx, M, vocab, off, N, hpn, b, reading="A"):
    ids = [int(v) for v in ids]
    req = [int(v) for v in req]
    local = [int(v) for v in local]
    ctx = [[int(v) for v in row] for row in ctx]
    M = [[int(v) for v in row] for row in M]
    vocab = [[int(v) for v in row] for row in vocab]
    off = [[int(v) for v in row] for row in off]
    T, L, C, H = len(ids), len(M), N - 1, (N - 1) * hpn
    out = [[[0] * H for _ in range(T)] for _ in range(L)]
    for t in range(T):
        q, r = local[t], req[t]

        def left(s):
            # the id s places left of token t
            if q >= s:
                return ids[t - s]
            return ctx[r][C + q - s]

        V = []
        for s in range(N):
            p = C + q
            valid = p - s >= 0 and all(left(d) != b for d in range(1, s + 1))
            if valid:
                V.append(left(s))
            else:
                V.append(b if reading == "A" else 0)
        for l in range(L):
            for n in range(2, N + 1):
                mix = 0
                for s in range(n):
                    mix ^= (V[s] * M[l][s]) & MASK
                mix = to_signed(mix)
                for j in range(hpn):
                    h = (n - 2) * hpn + j
                    out[l][t][h] = to_signed(mix % vocab[l][h] + off[l][h])
    return out
