"""Shared helpers of the GPU parity tests: device copies, poisoning, and the parity check against
the fp64 oracle (reference rounded to the output type, bound from the reduction length)."""
import numpy as np
import torch

from oracle import numerics

DEV = torch.device("cuda:0")


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage patterns of a CPU tensor (uint16 for 16-bit, uint8 for 8-bit types)."""
    t = t.contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def poisoned(shape, dtype) -> torch.Tensor:
    """A device tensor whose every byte is 0xFF (NaN in every float type used here)."""
    t = torch.empty(shape, dtype=dtype, device=DEV)
    t.view(torch.uint8).fill_(0xFF)
    return t


def unwritten_report(out: np.ndarray, limit: int = 8) -> str:
    """Rows (and the first columns) still holding the poison pattern, named, instead of a bare
    tolerance miss."""
    bad = ~np.isfinite(out)
    if not bad.any():
        return ""
    rows = np.unique(np.nonzero(bad.reshape(out.shape[0], -1))[0])
    return f"{int(bad.sum())} outputs unwritten or non-finite; rows {rows[:limit].tolist()}" \
           f"{' ...' if rows.size > limit else ''}"


_MBITS = {"f16": (10, -24), "bf16": (7, -133), "f32": (23, -149)}


def ulp(x: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of format ``fmt`` at |x| (the subnormal spacing below the normal range)."""
    mb, emin_sub = _MBITS[fmt]
    ax = np.maximum(np.abs(x), 2.0 ** (emin_sub + mb))
    e = np.floor(np.log2(ax))
    return np.exp2(np.maximum(e - mb, emin_sub))


def check_parity(out_dev: torch.Tensor, ref64: np.ndarray, out_dtype: str, kred: int,
                 kind: str = "16bit", what: str = ""):
    """Two checks. (1) The stated bound: max|out - round(ref)| <= 2e-2*sqrt(K/4096)*max|ref|
    (2e-2*max|ref| for fp8). (2) A much tighter one that fp32 accumulation always meets and a
    dropped or doubled partial never does: every element within one unit in the last place of
    the output type of the exact value, plus 1e-5*sqrt(K/4096)*max|ref| for the fp32 sums."""
    out = out_dev.float().cpu().double().numpy().reshape(ref64.shape)
    rep = unwritten_report(out)
    assert not rep, f"{what}: {rep}"
    ref = numerics.round_output(ref64, out_dtype)
    err = float(np.max(np.abs(out - ref))) if ref.size else 0.0
    tol = numerics.tolerance(ref, kred, kind)
    assert err <= tol, f"{what}: max|err| {err:.4e} > tol {tol:.4e}"
    if ref.size and np.max(np.abs(ref)) > 0:
        assert np.max(np.abs(out)) > 0, f"{what}: output is all zeros"
        amax = float(np.max(np.abs(ref64)))
        slack = ulp(ref64, out_dtype) + 1e-5 * np.sqrt(max(kred, 1) / 4096.0) * amax
        excess = np.abs(out - ref64) - slack
        worst = int(np.argmax(excess))
        assert excess.flat[worst] <= 0, (
            f"{what}: element {np.unravel_index(worst, ref64.shape)} = {out.flat[worst]!r}, exact "
            f"{ref64.flat[worst]!r}: off by more than one ulp + fp32 accumulation slack")
    return err, tol


def sample_points(M, N, n_random=2048, seed=0, tile=128):
    """Rows/cols at every tile edge plus random interior points; returns flat (ms, ns)."""
    rng = np.random.default_rng(seed)
    edge_r = sorted({x for t in range(0, M, tile) for x in (t, min(M - 1, t + tile - 1))})
    edge_c = sorted({x for t in range(0, N, tile) for x in (t, min(N - 1, t + tile - 1))})
    rr = rng.integers(0, M, size=64)
    cc = rng.integers(0, N, size=64)
    ms1, ns1 = np.meshgrid(np.array(edge_r), cc, indexing="ij")
    ms2, ns2 = np.meshgrid(rr, np.array(edge_c), indexing="ij")
    ms3 = rng.integers(0, M, size=n_random)
    ns3 = rng.integers(0, N, size=n_random)
    ms = np.concatenate([ms1.ravel(), ms2.ravel(), ms3])
    ns = np.concatenate([ns1.ravel(), ns2.ravel(), ns3])
    return ms.astype(np.int64), ns.astype(np.int64)
