"""Helpers shared by the GPU tests: run the CUDA path, compare with the oracle."""

import numpy as np
import torch

import mla_speculative_decoding_gb300 as mv
import oracle

# Tolerances of the method's contract: bf16 out within 1e-2 + 1e-2*|ref|,
# fp32 lse within 1e-3 absolute. The relative Frobenius bound is a tighter
# self-imposed check (at long context the outputs are ~1e-2 in size, so the
# absolute floor alone would barely constrain them).
OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3
REL_FRO = 1e-2


_CONFIG_CACHE = {}


def config_cached(idx, placement="scattered"):
    """Read-only cache of the named workloads (generation of the large ones
    takes seconds)."""
    key = (idx, placement)
    if key not in _CONFIG_CACHE:
        from workloads import make_config
        _CONFIG_CACHE[key] = make_config(idx, placement=placement)
    return _CONFIG_CACHE[key]


def run_gpu(inp, flags=0, use_anc=True, nsplit=None, device="cuda"):
    d = mv.to_device(inp, device=device, nsplit=nsplit)
    d.build()
    if flags:
        d.partial(flags=flags, use_anc=use_anc)
        d.combine()
    else:
        d.attention(use_anc=use_anc)
    torch.cuda.synchronize()
    return d


def host_out(d):
    o = d.out.float().cpu().numpy().astype(np.float64).reshape(-1, 512)
    l = d.lse.cpu().numpy().astype(np.float64).reshape(-1)
    return o, l


def status(d):
    return int(d.status.cpu().item())


def sample_rows(inp, per_request=8, seed=0):
    rng = np.random.default_rng(seed)
    H, T = inp.num_heads, inp.T
    rows = []
    for b in range(inp.batch):
        picks = {(0, 0), (T - 1, H - 1), (T // 2, 0)}
        while len(picks) < per_request:
            picks.add((int(rng.integers(T)), int(rng.integers(H))))
        rows += [(b * T + t) * H + h for t, h in sorted(picks)]
    return np.array(rows, dtype=np.int64)


def compare(out, lse, ref_out, ref_lse, what=""):
    err = np.abs(out - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    worst = float((err - bound).max())
    assert worst <= 0, f"{what}: out beyond tolerance by {worst:.3g} (max err {err.max():.3g})"
    lerr = float(np.abs(lse - ref_lse).max())
    assert lerr <= LSE_ATOL, f"{what}: lse error {lerr:.3g}"
    fro = float(np.linalg.norm(out - ref_out) / max(np.linalg.norm(ref_out), 1e-30))
    assert fro <= REL_FRO, f"{what}: relative Frobenius error {fro:.3g}"
    return dict(max_abs=float(err.max()), lse_max=lerr, rel_fro=fro)


def oracle_ref(inp, rows=None):
    ip, ix, _ = oracle.build_meta(inp)
    return oracle.verify_attention(inp, ip, ix, rows=rows)
