"""How many bits the B300 FP8 tensor core keeps when it accumulates.

    python -m fp8_fine_grained_20_b300.accum_probe [--json]

The pages (why-be.why-be.co.kr post 55081) report that FP8 GEMM accumulation
on H800 keeps about 14 bits, with a relative error near 2% at K = 4096, and
promote partial sums to FP32 every 128 K for that reason.  This script
measures the same two things on B300 with fp8_mma_accumulation_probe (whole-K
accumulation in tensor memory, no promotion):

1. Swamping: a row holds one large product 2^8 and small products
   2^(8 - gap); the result shows, per gap, whether a small term survives the
   addition -- (a) inside one MMA instruction (k = 1), (b) in the next MMA
   instruction of the same 128-deep block (k = 32), (c) in the next block
   (k = 128), (d) 127 small terms spread over consecutive instructions.
   The largest gap at which the sum is exact gives the effective significand
   width.  Columns 0-127 read B = 1 everywhere (gaps 0-17); columns 128-255
   read B = 2^-8 at the small positions (gaps 8-25).
2. Long sums: random codes (N(0,1) values quantized with one scale per
   128-block, codes only) at K = 128 .. 16384; relative error of the
   tensor-memory accumulation against the exact sum, next to the same sum
   accumulated in FP32 in k order and the promoted GEMM of this library (FP32
   promotion every 128 K, unit scales).
"""
import argparse
import json
import sys

import numpy as np
import torch

import fp8_fine_grained_20_b300 as fg


def pow2_code(e):
    """E4M3 code of 2^e, -9 <= e <= 8 (subnormal below 2^-6)."""
    if e >= -6:
        return (e + 7) << 3
    return {-7: 0x04, -8: 0x02, -9: 0x01}[e]


def decode_table():
    t = np.zeros(256, np.float64)
    for c in range(256):
        e, m = (c >> 3) & 0xF, c & 7
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        t[c] = -v if c & 0x80 else v
    t[0x7F] = t[0xFF] = np.nan
    return t


def swamping(K=4096):
    A = np.zeros((128, K), np.uint8)
    B = np.zeros((256, K), np.uint8)
    B[:, :] = pow2_code(0)
    B[128:, 1:] = pow2_code(-8)
    modes = {0: [1], 1: [32], 2: [128], 3: list(range(32, 32 * 128, 32))}
    for m in range(128):
        mode, g = divmod(m, 32)
        A[m, 0] = pow2_code(8)
        if g <= 17:
            A[m, modes[mode]] = pow2_code(8 - g)
    D = fg.fp8_mma_accumulation_probe(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    D = D.cpu().numpy().astype(np.float64)
    names = {0: "same instruction", 1: "next instruction", 2: "next 128-block", 3: "127 terms, one per instruction"}
    res = {}
    for mode in range(4):
        kept = {}
        for g in range(18):
            m = mode * 32 + g
            nsmall = len(modes[mode])
            for half, extra in ((0, 0), (1, 8)):
                gap = g + extra
                exact = 2.0 ** 8 + nsmall * 2.0 ** (8 - gap)
                got = D[m, 0 if half == 0 else 128]
                kept[gap] = bool(got == np.float64(np.float32(exact)) and got != 2.0 ** 8)
        exact_gaps = [gp for gp in sorted(kept) if kept[gp]]
        res[names[mode]] = {"largest_gap_kept": max(exact_gaps) if exact_gaps else None,
                            "kept_by_gap": {str(k): v for k, v in sorted(kept.items())}}
    return res


def long_sums(Ks=(128, 1024, 4096, 16384), seed=0):
    tab = decode_table()
    rng = np.random.default_rng(seed)
    out = {}
    for K in Ks:
        def codes(rows):
            x = rng.standard_normal((rows, K)).astype(np.float32)
            s = np.abs(x.reshape(rows, K // 128, 128)).max(axis=2, keepdims=True) / np.float32(448.0)
            y = (x.reshape(rows, K // 128, 128) / s).reshape(rows, K)
            return torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        A, B = codes(128), codes(256)
        ref = tab[A] @ tab[B].T                                      # exact in float64
        D = fg.fp8_mma_accumulation_probe(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
        ones_a = torch.ones((K // 128, 128), dtype=torch.float32, device="cuda").t()
        ones_b = torch.ones((K // 128, 2), dtype=torch.float32, device="cuda")
        C = fg.fp8_gemm_blockscaled(torch.from_numpy(A).cuda(), ones_a, torch.from_numpy(B).cuda(), ones_b,
                                    fg.FP8_SB_BLOCK128x128, out=torch.empty((128, 256), dtype=torch.bfloat16,
                                                                            device="cuda"))
        torch.cuda.synchronize()
        D = D.cpu().numpy().astype(np.float64)
        C = C.float().cpu().numpy().astype(np.float64)
        f32 = np.zeros((128, 256), np.float32)
        pa, pb = tab[A].astype(np.float32), tab[B].astype(np.float32)
        for k in range(K):                                          # FP32 accumulation in k order
            f32 = f32 + np.outer(pa[:, k], pb[:, k]).astype(np.float32)
        f32 = f32.astype(np.float64)

        def err(x):
            d = np.abs(x - ref)
            big = np.abs(ref) > 0.1 * np.sqrt(np.mean(ref ** 2))
            return {"frobenius_rel": float(np.linalg.norm(x - ref) / np.linalg.norm(ref)),
                    "max_rel_where_ref_gt_0.1rms": float(np.max(d[big] / np.abs(ref[big]))),
                    "max_abs_over_rms": float(d.max() / np.sqrt(np.mean(ref ** 2)))}
        out[K] = {"tmem_accumulation": err(D), "fp32_sequential": err(f32),
                  "promoted_gemm_bf16_out": err(C)}
    return out


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--json", action="store_true")
    args = p.parse_args(argv)
    torch.cuda.set_device(0)
    fg.capi()
    res = {"swamping": swamping(), "long_sums": long_sums()}
    status = fg.fp8_get_device_status(reset=True)
    if status != 0:
        raise SystemExit("device status %d" % status)
    if args.json:
        print(json.dumps(res))
        return
    for name, r in res["swamping"].items():
        print("swamping, %-32s largest exact gap %s  (significand ~%s bits)"
              % (name, r["largest_gap_kept"], None if r["largest_gap_kept"] is None else r["largest_gap_kept"] + 1))
    for K, r in res["long_sums"].items():
        print("K=%-6d " % K + "  ".join("%s: frob %.2e max_rel %.2e" % (k, v["frobenius_rel"],
                                                                        v["max_rel_where_ref_gt_0.1rms"])
                                         for k, v in r.items()))


if __name__ == "__main__":
    sys.exit(main())
