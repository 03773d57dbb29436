"""FLOP accounting of one Muon step (measurement only).

Per matrix with short side m and long side n, one Newton-Schulz iteration
forms A = X X^T (m x m, K = n), A*A (m x m, K = m) and B*X (m x n, K = m).
The symmetric products are counted as one triangle (m^2 n and m^3 flops),
B*X densely (2 m^2 n), so the algorithmic count is ns*(3 m^2 n + m^3); the
dense-equivalent count is ns*(4 m^2 n + 2 m^3).
"""


def algorithmic_flops(shapes, ns_steps=5):
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        tot += ns_steps * (3 * m * m * n + m ** 3)
    return tot


def dense_flops(shapes, ns_steps=5):
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        tot += ns_steps * (4 * m * m * n + 2 * m ** 3)
    return tot


def apply_flops(shapes, ns_steps=5):
    """Flops of the B*X products alone (2 m^2 n per iteration)."""
    return sum(ns_steps * 2 * min(r, c) ** 2 * max(r, c) for r, c in shapes)


def elementwise_bytes(shapes):
    """Algorithmic HBM bytes of the momentum/normalise pass: read G and M,
    write M (fp32) and the fp16 iterate: 14 bytes per element."""
    return sum(14 * r * c for r, c in shapes)


def gram_windows(ns_steps, restarts=(2,), max_window=2):
    """Restart windows the Gram backend runs: the restart positions inside
    (0, ns_steps), each window longer than ``max_window`` steps split into
    ceil(len / max_window) windows as even as possible, longer ones first."""
    cuts = sorted({int(k) for k in restarts if 0 < int(k) < ns_steps})
    bounds = [0] + cuts + [ns_steps]
    out = []
    for i in range(len(bounds) - 1):
        a, b = bounds[i], bounds[i + 1]
        if b <= a:
            continue
        length = b - a
        parts = -(-length // max_window)
        for j in range(parts):
            w = length // parts + (1 if j < length % parts else 0)
            out.append((a, a + w))
            a += w
    return out


def gram_flops(shapes, ns_steps=5, restarts=(2,)):
    """Algorithmic flops of the Gram-space backend, symmetric products as one
    triangle.  Per restart window: X X^T (m^2 n) and a closing Q X (2 m^2 n);
    per step Z from R R (m^3), Q' = Z Q on all but the window's first step
    (m^3), R Z and Z (R Z) on all but its last (2 m^3).  Windows are at most
    two steps long, so five steps (with the default restart before the
    third, or none) run as windows of 2, 2 and 1 steps: 9 m^2 n + 11 m^3."""
    windows = gram_windows(ns_steps, restarts)
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        for start, end in windows:
            tot += 3 * m * m * n
            for k in range(start, end):
                tot += m ** 3
                if k > start:
                    tot += m ** 3
                if k < end - 1:
                    tot += 2 * m ** 3
    return tot
