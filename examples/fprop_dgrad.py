"""Quantise X, W and dY and run the fprop and dgrad GEMMs through the binding
(needs a B300 and the built library)."""
import torch
from nvfp4_precision_02_b300 import binding as nv


def main():
    x = torch.randn(4096, 8192, dtype=torch.bfloat16, device="cuda")
    w = torch.randn(6144, 8192, dtype=torch.bfloat16, device="cuda") * 0.02
    qx = nv.quantize_1d(x)                        # 1x16 blocks, RNE
    qw, qwt, _ = nv.quantize_2d(w)                # 16x16 tiles: W and W^T
    y = nv.gemm(qx, qw)                           # bf16 [4096, 6144] = X . W^T
    dy = torch.randn_like(y) * 1e-3
    qdy = nv.quantize_1d(dy, mode=nv.SR, seed=7)  # stochastic rounding
    dx = nv.gemm(qdy, qwt)                        # dgrad: bf16 [4096, 8192] = dY . W
    torch.cuda.synchronize()
    print(y.shape, dx.shape)


if __name__ == "__main__":
    main()
