"""The reading behind the strided data gradient, checked on the CPU: a stride-(sh, sw) data gradient
equals, phase by phase, a stride-1 correlation of dy with a subset of the filter taps. For the dx
pixels h = sh*i + a only the taps r = r0 + sh*t with r0 = (a + ph) mod sh reach them, and
dx[sh*i + a] = sum_t dy[i + q - t] * w[r0 + sh*t] with q = (a + ph - r0) / sh; the GPU path runs
each phase as a traversal with Rt taps and low padding Rt - 1 - q. Here that identity is assembled
with numpy over many small geometries and compared with the oracle's direct loops."""
import itertools

import numpy as np
import pytest
import torch

from oracle import numerics


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _phase_1d(X, R, sigma, pad, a):
    r0 = (a + pad) % sigma
    rt = (R - 1 - r0) // sigma + 1 if r0 < R else 0
    q = (a + pad - r0) // sigma
    xp = (X - 1 - a) // sigma + 1 if a < X else 0
    return xp, rt, r0, rt - 1 - q


def _by_phases(dy, w, H, W, stride, pad):
    """dx from one stride-1 correlation per output phase (one group)."""
    N, Ho, Wo, K = dy.shape
    _, R, S, C = w.shape
    sh, sw = stride
    dx = np.zeros((N, H, W, C))
    for a, b in itertools.product(range(sh), range(sw)):
        hp, rt, r0, padh = _phase_1d(H, R, sh, pad[0], a)
        wp, st, s0, padw = _phase_1d(W, S, sw, pad[1], b)
        if not (hp and wp and rt and st):
            continue                               # no tap reaches these pixels: they stay 0
        # dy padded so that the traversal window of pixel (i, j) starts at (i - padh, j - padw)
        lo_h, lo_w = max(padh, 0), max(padw, 0)
        pad_dy = np.zeros((N, Ho + 2 * lo_h + rt + hp, Wo + 2 * lo_w + st + wp, K))
        pad_dy[:, lo_h:lo_h + Ho, lo_w:lo_w + Wo] = dy
        for r, s in itertools.product(range(rt), range(st)):   # traversal offsets
            fr, fs = r0 + sh * (rt - 1 - r), s0 + sw * (st - 1 - s)
            h0, w0 = lo_h - padh + r, lo_w - padw + s
            win = pad_dy[:, h0:h0 + hp, w0:w0 + wp, :]          # [N, hp, wp, K]
            dx[:, a::sh, b::sw, :][:, :hp, :wp, :] += win @ w[:, fr, fs, :]
    return dx


GEOMS = [(H, W, R, S, sh, sw, ph, pw)
         for (H, W) in [(7, 9), (8, 8), (5, 11)]
         for (R, S) in [(1, 1), (3, 3), (3, 2), (4, 1)]
         for (sh, sw) in [(2, 2), (3, 1), (2, 4)]
         for (ph, pw) in [(0, 0), (R - 1, S - 1), ((R - 1) // 2, 0)]
         if H + 2 * ph >= R and W + 2 * pw >= S]


@pytest.mark.parametrize("H,W,R,S,sh,sw,ph,pw", GEOMS)
def test_phase_decomposition_equals_the_direct_data_gradient(H, W, R, S, sh, sw, ph, pw):
    Ho, Wo = (H + 2 * ph - R) // sh + 1, (W + 2 * pw - S) // sw + 1
    g = torch.Generator().manual_seed(H * 1000 + W * 100 + R * 10 + S + sh * 7 + sw * 3 + ph + pw)
    dy = (torch.rand((2, Ho, Wo, 8), generator=g) * 2 - 1).to(torch.float16)
    w = (torch.rand((8, R, S, 8), generator=g) * 2 - 1).to(torch.float16)
    ref = numerics.dgrad_nhwc("f16", _bits(dy), _bits(w), H, W, (sh, sw), (ph, pw), 1)
    got = _by_phases(dy.double().numpy(), w.double().numpy(), H, W, (sh, sw), (ph, pw))
    np.testing.assert_allclose(got.reshape(-1, 8), ref, rtol=1e-12, atol=1e-12)


def test_phases_partition_the_pixels_and_taps():
    # every dx pixel lies in exactly one phase, and every (pixel, tap) pair that the definition
    # sums over is covered once by its phase's tap set
    for H, R, sigma, pad in itertools.product(range(1, 12), range(1, 6), range(1, 5), range(0, 5)):
        if pad >= R:
            continue
        seen = 0
        for a in range(sigma):
            xp, rt, r0, _ = _phase_1d(H, R, sigma, pad, a)
            seen += xp
            taps = {r0 + sigma * t for t in range(rt)}
            assert taps == {r for r in range(R) if (a + pad - r) % sigma == 0}
        assert seen == H
