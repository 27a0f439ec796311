"""Small cases over every kernel of the library, for the bounds-checked
build: each call's outputs (as numpy arrays) and the device status after it.
Run in a process whose ops module loaded either build of the library."""
import numpy as np
import torch

from quantised_linear_layers_gb300 import synthetic as syn


def _np(t):
    t = t.detach()
    if t.dtype in (torch.float8_e4m3fn,):
        t = t.view(torch.uint8)
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy().copy()


def run(ops):
    """Returns {case name: (list of output arrays, device status after it)}."""
    out = {}
    dev = "cuda"

    def rec(name, tensors):
        torch.cuda.synchronize()
        out[name] = ([_np(t) for t in tensors], ops.device_status())

    x = syn.randn_row_exp(300, 520, dtype=torch.bfloat16).to(dev)
    xf = syn.randn_row_exp(130, 200, dtype=torch.float32).to(dev)
    for fmt in (0, 1, 2):
        for gran in (32, 128):
            rec(f"token_rows_f{fmt}_g{gran}", ops.fp8_cast_per_token(x, gran, fmt))
            rec(f"token_rows_f32_f{fmt}_g{gran}", ops.fp8_cast_per_token(xf, gran, fmt))
            rec(f"token_cols_f{fmt}_g{gran}", ops.fp8_cast_per_token(x.t(), gran, fmt))               # TMA-staged
            rec(f"token_cols_unal_f{fmt}_g{gran}", ops.fp8_cast_per_token(x[:, 1:].t(), gran, fmt))  # unaligned
            xc = x.t().contiguous().t()
            rec(f"token_colmajor_f{fmt}_g{gran}", ops.fp8_cast_per_token(xc, gran, fmt, out=torch.empty_like(
                xc, dtype=torch.float8_e4m3fn).t().contiguous().t()))
            rec(f"token_generic_f{fmt}_g{gran}", ops.fp8_cast_per_token(x[::2, ::3], gran, fmt))
        rec(f"dual_token_f{fmt}", ops.fp8_cast_per_token_dual(x, fmt))
        rec(f"block_f{fmt}", ops.fp8_cast_per_block(x, fmt))
        rec(f"block_t_f{fmt}", ops.fp8_cast_per_block(x.t(), fmt))
        rec(f"block_dual_f{fmt}", ops.fp8_cast_per_block_dual(x, fmt))

    rec("token_recip_g128", ops.fp8_cast_per_token(x, 128, 0, recip=True))
    rec("block_recip", ops.fp8_cast_per_block(x, 0, recip=True))

    # GEMMs: every path
    m, n, k = 300, 520, 640
    a = syn.randn((m, k), seed=61).to(dev)
    w = syn.randn((n, k), seed=62, mul=0.02).to(dev)
    for fmt, paths in ((0, (0, 5, 6, 7)), (2, (0, 1, 2, 3, 4, 7))):
        aq, sa = ops.fp8_cast_per_token(a, 128, fmt, sf_mn_major=True)
        wq, sw = ops.fp8_cast_per_block(w, fmt)
        for path in paths:
            ops.set_gemm_path(path)
            try:
                rec(f"gemm_f{fmt}_p{path}", [ops.gemm_fp8_nt_bf16(aq, sa, wq, sw, fmt)])
                d0 = syn.randn((m, n), seed=63, dtype=torch.float32).to(dev)
                bq, sb = ops.fp8_cast_per_token(w, 128, fmt)
                d = d0.clone()
                ops.gemm_fp8_wgrad_fp32(aq, sa, bq, sb, out=d, accumulate=True, fmt=fmt)
                rec(f"wgrad_acc_f{fmt}_p{path}", [d])
                if path in (0, 1, 3):
                    rec(f"fp8out_f{fmt}_p{path}", ops.gemm_fp8_nt_fp8out(aq, sa, wq, sw, fmt, 128, 2))
            finally:
                ops.set_gemm_path(0)
        # MN-major operands (weight gradient and data gradient)
        t_, c1, c2 = 384, 260, 200
        dy = syn.randn((t_, c1), seed=64).to(dev)
        xx = syn.randn((t_, c2), seed=65).to(dev)
        dq, ds, dcq, dcs = ops.fp8_cast_per_token_dual(dy, fmt)
        xq, xs, xcq, xcs = ops.fp8_cast_per_token_dual(xx, fmt)
        rec(f"wgrad_mn_f{fmt}", [ops.gemm_fp8_wgrad_fp32_mn(dcq, dcs, xcq, xcs, fmt=fmt)])
        w2 = syn.randn((c1, c2), seed=66, mul=0.02).to(dev)
        w2q, w2s, w2st = ops.fp8_cast_per_block_dual(w2, fmt)
        rec(f"dgrad_nn_f{fmt}", [ops.gemm_fp8_nn_bf16(dq, ds, w2q, w2st, fmt)])
    # edges, at shapes the parity tests also run: one row, one column, cut
    # groups and tiles in both directions; split-K with a single row
    for shape in ((1, 512), (509, 1), (7, 33), (1, 24), (130, 36), (1, 130)):
        xe = syn.randn_row_exp(*shape, dtype=torch.bfloat16).to(dev)
        tag = f"{shape[0]}x{shape[1]}"
        for fmt in (0, 2):
            rec(f"edge_rows_{tag}_f{fmt}", ops.fp8_cast_per_token(xe, 32, fmt))
            rec(f"edge_t_{tag}_f{fmt}", ops.fp8_cast_per_token(xe.t(), 128, fmt))
            rec(f"edge_dual_{tag}_f{fmt}", ops.fp8_cast_per_token_dual(xe, fmt))
            rec(f"edge_block_dual_{tag}_f{fmt}", ops.fp8_cast_per_block_dual(xe, fmt))
    a1 = syn.randn((1, 4096), seed=71).to(dev)
    w1 = syn.randn((512, 4096), seed=72, mul=0.02).to(dev)
    for fmt, paths in ((0, (0, 7)), (2, (0, 4, 7))):
        a1q, a1s = ops.fp8_cast_per_token(a1, 128, fmt, sf_mn_major=True)
        w1q, w1s = ops.fp8_cast_per_block(w1, fmt)
        for path in paths:
            ops.set_gemm_path(path)
            try:
                rec(f"splitk_1x512x4096_f{fmt}_p{path}", [ops.gemm_fp8_nt_bf16(a1q, a1s, w1q, w1s, fmt)])
            finally:
                ops.set_gemm_path(0)
    # grouped GEMM (4 experts, padding rows)
    tokens = [128, 96, 112, 144]
    idx, _ = syn.contiguous_layout(tokens, 128)
    mg = idx.numel()
    ag = syn.randn((mg, 512), seed=67).to(dev)
    agq, ags = ops.fp8_cast_per_token(ag, 128, 2, sf_mn_major=True)
    wg = torch.empty((4, 256, 512), dtype=torch.float8_e4m3fn, device=dev)
    wgs = torch.empty((4, 2, 1), dtype=torch.int32, device=dev)
    for e in range(4):
        ops.fp8_cast_per_block(syn.randn((256, 512), seed=70 + e, mul=0.02).to(dev), 2, out=wg[e], out_sf=wgs[e])
    dg = torch.zeros((mg, 256), dtype=torch.bfloat16, device=dev)
    ops.m_grouped_gemm_fp8_nt_bf16_contiguous(agq, ags, wg, wgs, idx.to(dev), 2, out=dg)
    rec("grouped", [dg])
    # host-buffer pipeline
    xh = syn.randn((300, 512), seed=68).pin_memory()
    wq3, ws3 = ops.fp8_cast_per_block(syn.randn((256, 512), seed=69, mul=0.02).to(dev), 2)
    oh = torch.zeros((300, 256), dtype=torch.bfloat16).pin_memory()
    wsp = torch.empty(ops.cast_gemm_host_workspace_size(256, 512, 128, 2), dtype=torch.uint8, device=dev)
    ops.cast_gemm_host(xh, wq3, ws3, 2, oh, 128, wsp)
    rec("host_pipeline", [oh])
    return out


if __name__ == "__main__":
    import sys
    from quantised_linear_layers_gb300 import ops
    res = run(ops)
    arrays = {}
    for name, (arrs, st) in res.items():
        arrays[f"{name}__status"] = np.array([st])
        for i, arr in enumerate(arrs):
            arrays[f"{name}__{i}"] = arr
    np.savez(sys.argv[1], **arrays)
    print("flag", int(ops.load_library().ql_bounds_checked()))
