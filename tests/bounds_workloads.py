"""Runs one call of every kernel path on fixed seeded inputs and saves the outputs (npz),
with the library that VQ3_LIB selects. The bounds-check test runs it twice: once with the
bounds-check build (libvq3_bc.so), whose skipped-access counts go into the npz as
`bounds_<file>`, and once with the normal build; the outputs must agree bit for bit and
every count must be zero.

    VQ3_LIB=.../libvq3_bc.so python -m tests.bounds_workloads out.npz
"""

import sys

import numpy as np
import torch

from synth import inputs as S

DEV = "cuda"


def _f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(DEV)


def run(vq3) -> dict[str, np.ndarray]:
    out: dict[str, np.ndarray] = {}

    def keep(name, t):
        torch.cuda.synchronize()
        out[name] = t.detach().cpu().numpy().copy()

    # SwiGLU block at 5120 / 17408 with sign vectors: decode (1, 8, 16 rows), the prefill GEMM
    # up to 128 rows (64) and above (300)
    wl = S.mlp_27b(seed=40, rows=300)
    blk = S.add_signs(S.rng(40, 2), wl.layers[0])
    layer = vq3.MLP.from_block(blk, DEV)
    for rows in (1, 8, 16, 64, 300):
        keep(f"mlp_T{rows}", vq3.mlp_forward(_f16(wl.x[:rows]), layer))
    # the pre-norm residual step (residual add, sums of squares, RMSNorm inside the decode kernel)
    r = _f16(wl.x[:8])
    o = torch.empty_like(r)
    rn = torch.empty_like(r)
    ssn = torch.empty((8, 5120 // 16), dtype=torch.float32, device=DEV)
    vq3.mlp_prenorm_step(r, layer, o, rn, ss_next=ssn)
    keep("prenorm_out", o)
    keep("prenorm_r_next", rn)
    keep("prenorm_ss_next", ssn)
    d = _f16(S.activations(S.rng(41, 0), 8, 5120))
    ro = torch.empty_like(r)
    o2 = torch.empty_like(r)
    vq3.mlp_forward_residual(r, d, layer, ro, o2)
    keep("residual_r_out", ro)
    keep("residual_out", o2)
    keep("rmsnorm", vq3.residual_rmsnorm(r, d))

    # a 5120 -> 6144 linear with rank-64 factors: fused decode (1, 8) and the factor kernels (64, 300)
    m = S.matrix(S.rng(42), 5120, 6144, 1024, "2x16")
    m.signs = S.sign_bits(S.rng(42, 2), 5120)
    S.add_lowrank(S.rng(42, 3), m, 64, 0.02)
    lin = vq3.Linear.from_matrix(m, DEV)
    x = S.activations(S.rng(42, 0), 300, 5120)
    for rows in (1, 8, 64, 300):
        keep(f"linear_lr_T{rows}", vq3.linear_forward(_f16(x[:rows]), lin))

    # rotation alone, in both output orders
    keep("fwht", vq3.fwht_rotate(_f16(x[:3]), 1024, torch.from_numpy(m.signs.view(np.int32)).to(DEV)))

    # delta rule: the tensor-core kernel (d_k 128, a ragged last block) and the CUDA-core one (d_k 24)
    for dk, tokens in ((128, 13), (24, 13)):
        inp = S.delta_rule_inputs(seed=43, tokens=tokens, heads=4, d_k=dk, d_v=64)
        st = torch.from_numpy(inp.state).to(DEV)
        y = vq3.delta_rule_forward(_f16(inp.q), _f16(inp.k), _f16(inp.v), torch.from_numpy(inp.beta).to(DEV),
                                   torch.from_numpy(inp.alpha).to(DEV), st)
        keep(f"delta_dk{dk}", y)
        keep(f"delta_dk{dk}_state", st)
    return out


def main(path: str) -> None:
    from bit_vector_lut_gb300 import vq3
    out = run(vq3)
    try:
        for name, (count, site) in vq3.bounds_check(reset=True).items():
            out[f"bounds_{name}"] = np.array([count, site], dtype=np.int64)
    except vq3.Vq3Error:
        pass  # the normal build records nothing
    out["version"] = np.array(vq3.version())
    np.savez(path, **out)


if __name__ == "__main__":
    main(sys.argv[1])
