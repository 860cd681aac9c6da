"""Full-size acceptance of the block-scaled GEMMs against the FP64 oracle on
EVERY output element (the parity tests check these workloads on sampled
outputs only).

    python tests/full_oracle_acceptance.py [--out FILE] [--only NAME ...]

For each workload the inputs come from the seeded generators, the ORACLE
quantizes them (so the GEMM is tested in isolation), the library computes the
GEMM on the GPU, and the whole output is compared with the oracle's dense
FP64 product of the dequantized operands (oracle.gemm_blockscaled_dense,
reading R6), element by element, against the acceptance bound
|got - ref| <= 2^-7 |ref| + 1e-4 rms(ref), plus the relative Frobenius error
<= 5e-3.  Workloads: forward [8192 x 18432, K 7168], weight gradient
[7168 x 18432, K 8192 tokens], data gradient [8192 x 7168, K 18432], the MoE
grouped GEMM (32 experts [7168 x 2048], 16384 tokens x 8, Zipf 1.1), and the
same four with power-of-two scales through the hardware-scaled (MX) GEMMs.
The largest per-element ratio of the error to the bound, the Frobenius
error and the count of violations are printed as one JSON object per
workload.  Needs a CUDA GPU and a few minutes of host FP64 matmul.
"""
import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import fp8_fine_grained_20_b300 as fg  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

T, CIN, COUT = 8192, 7168, 18432
REL_TOL, ABS_TOL_RMS, FROB_TOL = 2.0 ** -7, 1e-4, 5e-3


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def mn(s):
    """Logical [R, C] fp32 scales on the device, stride 1 along R."""
    return dev(np.ascontiguousarray(s.T)).t()


def compare(name, got, ref, seconds):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    bound = REL_TOL * np.abs(ref) + ABS_TOL_RMS * rms
    ratio = err / bound
    frob = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    res = {"workload": name, "outputs": int(ref.size), "max_error_over_bound": float(ratio.max()),
           "violations": int((ratio > 1.0).sum()), "rel_frobenius": frob,
           "pass": bool((ratio <= 1.0).all() and frob <= FROB_TOL and np.isfinite(got).all()),
           "host_seconds": round(seconds, 1)}
    print(json.dumps(res), flush=True)
    return res


def gemm_case(name, qa, sa, qbt, sb, sb_kind, mx):
    t0 = time.time()
    f = fg.fp8_gemm_blockscaled_mx if mx else fg.fp8_gemm_blockscaled
    C = f(dev(qa), mn(sa), dev(qbt), dev(sb), sb_kind)
    torch.cuda.synchronize()
    got = C.float().cpu().numpy().astype(np.float64)
    del C
    kind = oracle.SB_COL128x1 if sb_kind == fg.FP8_SB_COL128x1 else oracle.SB_BLOCK128x128
    ref = oracle.gemm_blockscaled_dense(qa, sa, qbt, sb, kind)
    return compare(name, got, ref, time.time() - t0)


def forward(mx, th):
    x, _ = synth.activation(3, T, CIN, outlier_frac=0.0)
    w = synth.weight(3, CIN, COUT)
    qa, sa = oracle.quant_act_1x128(x, threads=th, pow2=mx)
    qw, sw = oracle.quant_w_128x128(w, threads=th, pow2=mx)
    return gemm_case("forward" + ("_mx" if mx else ""), qa, sa, np.ascontiguousarray(qw.T), sw,
                     fg.FP8_SB_BLOCK128x128, mx)


def weight_gradient(mx, th):
    x = synth.wgrad_tensor(4, 0, T, CIN)
    dy = synth.wgrad_tensor(4, 1, T, COUT)
    qx, sx = oracle.requant_1x128_to_128x1(*oracle.quant_act_1x128(x, threads=th, pow2=mx), threads=th, pow2=mx)
    qd, sd = oracle.requant_1x128_to_128x1(*oracle.quant_act_1x128(dy, threads=th, pow2=mx), threads=th, pow2=mx)
    return gemm_case("weight_gradient" + ("_mx" if mx else ""), qx, sx, qd, np.ascontiguousarray(sd.T),
                     fg.FP8_SB_COL128x1, mx)


def data_gradient(mx, th):
    dy = synth.wgrad_tensor(6, 1, T, COUT)
    w = synth.weight(6, CIN, COUT)
    qa, sa = oracle.quant_act_1x128(dy, threads=th, pow2=mx)
    qw, sw = oracle.quant_w_128x128(w, threads=th, pow2=mx)       # forward layout [Cin, Cout]: K-major B
    sbT = np.ascontiguousarray(sw.T)                                # logical [K/128 = Cout/128, N/128 = Cin/128]
    return gemm_case("data_gradient" + ("_mx" if mx else ""), qa, sa, qw, sbT, fg.FP8_SB_BLOCK128x128, mx)


def moe(mx, th):
    t0 = time.time()
    inp = synth.moe_inputs(seed=5)
    G, K, N = inp.w.shape
    qa, sa = oracle.quant_act_1x128(inp.x, threads=th, pow2=mx)
    qb = np.empty((G, N, K), np.uint8)
    sb = np.empty((G, K // 128, N // 128), np.float32)
    for g in range(G):
        qw, sw = oracle.quant_w_128x128(inp.w[g], threads=th, pow2=mx)
        qb[g] = qw.T
        sb[g] = sw
    f = fg.fp8_grouped_gemm_blockscaled_mx if mx else fg.fp8_grouped_gemm_blockscaled
    C = f(dev(qa), mn(sa), dev(qb), dev(sb), dev(inp.offsets))
    torch.cuda.synchronize()
    got_all = C.float().cpu().numpy().astype(np.float64)
    del C
    gots, refs = [], []
    for g in range(G):
        r0, r1 = int(inp.offsets[g]), int(inp.offsets[g + 1])
        if r1 > r0:   # routed rows and pad rows (zero codes, zero scales: exact zeros)
            refs.append(oracle.gemm_blockscaled_dense(qa[r0:r1], sa[r0:r1], qb[g], sb[g]))
            gots.append(got_all[r0:r1])
    return compare("moe_grouped" + ("_mx" if mx else ""), np.concatenate(gots), np.concatenate(refs),
                   time.time() - t0)


CASES = {"forward": forward, "weight_gradient": weight_gradient, "data_gradient": data_gradient, "moe": moe}


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--out", default=None, help="also write the results as a JSON list")
    p.add_argument("--only", nargs="*", default=None, choices=sorted(CASES))
    args = p.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("needs a CUDA GPU")
    torch.cuda.set_device(0)
    th = oracle.default_threads()
    results = []
    for mx in (False, True):
        for name, fn in CASES.items():
            if args.only and name not in args.only:
                continue
            results.append(fn(mx, th))
            torch.cuda.empty_cache()
    status = fg.fp8_get_device_status(reset=True)
    if args.out:
        with open(args.out, "w") as f:
            json.dump({"results": results, "device_status": status, "host_threads": th}, f, indent=1)
    return 0 if all(r["pass"] for r in results) and status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
