"""One kernel of the FP8 path at its benchmark size, for profiler captures.

    python profile_case.py KERNEL [--launches N] [--warmup W]

KERNEL is one of quant_act, quant_w, quant_w_moe (32 experts in one batched
launch), requant, gemm_fprop, gemm_fprop_q (the forward GEMM with the 1x128
quantizing epilogue), gemm_dgrad, gemm_wgrad, grouped_gemm, the power-of-two
GEMMs whose scales the tensor core applies (gemm_fprop_mx, gemm_wgrad_mx,
grouped_gemm_mx) and swiglu (SwiGLU recompute + 1x128 quantization of
cached gate/up [8192, 2 x 18432]).  The process allocates only what that one call needs (at most
about 2 GB), fills the bf16 inputs on the device with torch's generator
(N(0,1) activations with 1% of channels x100, N(0, 0.02^2) weights,
N(0, 1e-3^2) gradients), quantizes them with the library where the kernel
takes FP8 operands, then launches the kernel W + N times.  Under
``ncu -k regex:<name> -s W -c N`` only the last N launches are captured; the
setup kernels are not.

Kernel names to filter on: k_quant_act_1x128, k_quant_w_128x128,
k_requant_1x128_to_128x1, k_gemm_blockscaled, k_gemm_mx, k_swiglu_quant_1x128.
"""
import argparse
import os
import sys

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import torch  # noqa: E402

import fp8_fine_grained_20_b300 as fg  # noqa: E402

T, CIN, COUT = 8192, 7168, 18432
G, MOE_K, MOE_N, TOKENS, TOPK, ZIPF = 32, 7168, 2048, 16384, 8, 1.1


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def activation(rows, cols, seed):
    g = _gen(seed)
    idx = torch.randperm(cols, generator=g, device="cuda")[:round(0.01 * cols)]
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, rows, 8192):       # fp32 temporaries of at most 8192 rows
        x = torch.randn((min(8192, rows - r0), cols), generator=g, device="cuda", dtype=torch.float32)
        x[:, idx] *= 100.0
        out[r0:r0 + x.shape[0]] = x.to(torch.bfloat16)
    return out


def weight(rows, cols, seed, sigma=0.02):
    g = _gen(seed)
    return (torch.randn((rows, cols), generator=g, device="cuda", dtype=torch.float32) * sigma).to(torch.bfloat16)


def moe_offsets(seed):
    """Padded per-expert row ranges of the benchmark's MoE workload (the seeded
    routing of the `synth` input module: 16384 tokens x 8 picks, p_g ~ (g+1)^-1.1)."""
    import synth
    _, offsets = synth.moe_routing(seed, G, TOKENS, TOPK, ZIPF)
    return torch.from_numpy(offsets)


def setup(kind):
    """Returns a closure that launches the kernel once."""
    if kind == "quant_act":
        x = activation(T, CIN, 1)
        q = torch.empty((T, CIN), dtype=torch.uint8, device="cuda")
        s = torch.empty((CIN // 128, T), dtype=torch.float32, device="cuda").t()
        return lambda: fg.fp8_quant_act_1x128(x, q, s)
    if kind == "quant_w":
        w = weight(CIN, COUT, 2)
        q = torch.empty((COUT, CIN), dtype=torch.uint8, device="cuda")
        s = torch.empty((CIN // 128, COUT // 128), dtype=torch.float32, device="cuda")
        return lambda: fg.fp8_quant_w_128x128(w, q, s)
    if kind == "quant_w_moe":
        w = weight(G * MOE_K, MOE_N, 10).view(G, MOE_K, MOE_N)
        q = torch.empty((G, MOE_N, MOE_K), dtype=torch.uint8, device="cuda")
        s = torch.empty((G, MOE_K // 128, MOE_N // 128), dtype=torch.float32, device="cuda")
        return lambda: fg.fp8_quant_w_128x128_batched(w, q, s)
    if kind == "requant":
        q, s = fg.fp8_quant_act_1x128(activation(T, CIN, 3))
        qT = torch.empty((CIN, T), dtype=torch.uint8, device="cuda")
        sT = torch.empty((T // 128, CIN), dtype=torch.float32, device="cuda").t()
        return lambda: fg.fp8_requant_1x128_to_128x1(q, s, qT, sT)
    if kind == "gemm_fprop":
        a, sa = fg.fp8_quant_act_1x128(activation(T, CIN, 4))
        b, sb = fg.fp8_quant_w_128x128(weight(CIN, COUT, 5))
        c = torch.empty((T, COUT), dtype=torch.bfloat16, device="cuda")
        return lambda: fg.fp8_gemm_blockscaled(a, sa, b, sb, fg.FP8_SB_BLOCK128x128, c)
    if kind == "gemm_fprop_q":
        a, sa = fg.fp8_quant_act_1x128(activation(T, CIN, 4))
        b, sb = fg.fp8_quant_w_128x128(weight(CIN, COUT, 5))
        q = torch.empty((T, COUT), dtype=torch.uint8, device="cuda")
        s = torch.empty((COUT // 128, T), dtype=torch.float32, device="cuda").t()
        return lambda: fg.fp8_gemm_blockscaled_q1x128(a, sa, b, sb, fg.FP8_SB_BLOCK128x128, q, s)
    if kind == "gemm_dgrad":
        a, sa = fg.fp8_quant_act_1x128(weight(T, COUT, 11, 1e-3))
        b, sb = fg.fp8_quant_w_128x128(weight(CIN, COUT, 12), q_layout=fg.FP8_ROWMAJOR_KN)
        c = torch.empty((T, CIN), dtype=torch.bfloat16, device="cuda")
        return lambda: fg.fp8_gemm_blockscaled(a, sa, b, sb.t(), fg.FP8_SB_BLOCK128x128, c)
    if kind == "gemm_wgrad":
        xq, xs = fg.fp8_quant_act_1x128(weight(T, CIN, 6, 1e-3))
        dq, ds = fg.fp8_quant_act_1x128(weight(T, COUT, 7, 1e-3))
        a, sa = fg.fp8_requant_1x128_to_128x1(xq, xs)
        b, sb = fg.fp8_requant_1x128_to_128x1(dq, ds)
        del xq, xs, dq, ds
        c = torch.empty((CIN, COUT), dtype=torch.bfloat16, device="cuda")
        return lambda: fg.fp8_gemm_blockscaled(a, sa, b, sb.t(), fg.FP8_SB_COL128x1, c)
    if kind == "grouped_gemm":
        off = moe_offsets(5)
        rows = int(off[-1])
        a, sa = fg.fp8_quant_act_1x128(activation(rows, MOE_K, 9))
        bq, bs = fg.fp8_quant_w_128x128_batched(weight(G * MOE_K, MOE_N, 100).view(G, MOE_K, MOE_N))
        c = torch.empty((rows, MOE_N), dtype=torch.bfloat16, device="cuda")
        d_off = off.cuda()
        return lambda: fg.fp8_grouped_gemm_blockscaled(a, sa, bq, bs, d_off, c)
    if kind == "gemm_fprop_mx":
        a, sa = fg.fp8_quant_act_1x128_pow2(activation(T, CIN, 4))
        b, sb = fg.fp8_quant_w_128x128_pow2(weight(CIN, COUT, 5))
        c = torch.empty((T, COUT), dtype=torch.bfloat16, device="cuda")
        return lambda: fg.fp8_gemm_blockscaled_mx(a, sa, b, sb, fg.FP8_SB_BLOCK128x128, c)
    if kind == "gemm_wgrad_mx":
        xq, xs = fg.fp8_quant_act_1x128_pow2(weight(T, CIN, 6, 1e-3))
        dq, ds = fg.fp8_quant_act_1x128_pow2(weight(T, COUT, 7, 1e-3))
        a, sa = fg.fp8_requant_1x128_to_128x1_pow2(xq, xs)
        b, sb = fg.fp8_requant_1x128_to_128x1_pow2(dq, ds)
        del xq, xs, dq, ds
        c = torch.empty((CIN, COUT), dtype=torch.bfloat16, device="cuda")
        return lambda: fg.fp8_gemm_blockscaled_mx(a, sa, b, sb.t(), fg.FP8_SB_COL128x1, c)
    if kind == "grouped_gemm_mx":
        off = moe_offsets(5)
        rows = int(off[-1])
        a, sa = fg.fp8_quant_act_1x128_pow2(activation(rows, MOE_K, 9))
        bq, bs = fg.fp8_quant_w_128x128_batched_pow2(weight(G * MOE_K, MOE_N, 100).view(G, MOE_K, MOE_N))
        c = torch.empty((rows, MOE_N), dtype=torch.bfloat16, device="cuda")
        d_off = off.cuda()
        return lambda: fg.fp8_grouped_gemm_blockscaled_mx(a, sa, bq, bs, d_off, c)
    if kind == "swiglu":
        gu = weight(T, 2 * COUT, 13, 1.7)
        q = torch.empty((T, COUT), dtype=torch.uint8, device="cuda")
        s = torch.empty((COUT // 128, T), dtype=torch.float32, device="cuda").t()
        return lambda: fg.fp8_swiglu_quant_1x128(gu, q=q, s=s)
    raise SystemExit("unknown kernel %r" % kind)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("kernel", choices=["quant_act", "quant_w", "quant_w_moe", "requant", "gemm_fprop",
                                      "gemm_fprop_q", "gemm_dgrad", "gemm_wgrad", "grouped_gemm",
                                      "gemm_fprop_mx", "gemm_wgrad_mx", "grouped_gemm_mx", "swiglu"])
    p.add_argument("--launches", type=int, default=1)
    p.add_argument("--warmup", type=int, default=2)
    args = p.parse_args(argv)
    torch.cuda.set_device(0)
    fg.capi()
    run = setup(args.kernel)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()    # release the generators' fp32 temporaries before any capture
    for _ in range(args.warmup + args.launches):
        run()
    torch.cuda.synchronize()
    status = fg.fp8_get_device_status(reset=True)
    if status != 0:
        raise SystemExit("device status %d" % status)
    print("%s: %d launches ok" % (args.kernel, args.warmup + args.launches))


if __name__ == "__main__":
    sys.exit(main())
