"""The backward parity checks shared by the BF16 and MXFP8 GPU tests.

Step by step, on what the GPU produced:
  * the saved pre-activations A against the oracle's bf16(W13 x): bit-exact except flagged
    roundings;
  * dA and w*h (and, in MXFP8, dA's codes and scales) from the GPU's own A;
  * dx from the GPU's own dA (MXFP8: its dequantized dA codes), dW13 and dW2 from the GPU's
    own dA and w*h;
  * d_topk_w from the GPU's own A, d_logits from the GPU's own d_topk_w;
and end to end from the layer's inputs within the stated tolerance.
"""
import numpy as np

import oracle
from harness import (TOL_BF16, TOL_MXFP8, check_codes, check_exact, check_tol, host,
                     padded_rows, preact_rows, remap_experts, sorted_rows)
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import workspace_item


def gpu_state(L, ws, which, pre):
    """Host copies of what the checks read from the GPU: schedule, padded offsets, saved A,
    dA, w*h (and MXFP8 dA codes and scales)."""
    import torch
    T, I, K, E = L.T, L.I, L.K, L.E
    R = T * K
    st = dict(
        perm=L.sched.perm[:R].cpu().numpy(), inv=L.sched.inv[:R].cpu().numpy(),
        offsets=L.sched.offsets[:E + 1].cpu().numpy(),
        poff=workspace_item(ws, L.cfg, which, B.MOK_ITEM_PAD_OFFSETS).view(torch.int32)
        .cpu().numpy(),
        pre=pre[:R],
        dA=workspace_item(ws, L.cfg, which, B.MOK_ITEM_DA).view(torch.bfloat16).view(-1, 2 * I),
        sh=workspace_item(ws, L.cfg, which, B.MOK_ITEM_WH).view(torch.bfloat16).view(-1, I))
    if L.cfg.prec == B.MOK_MXFP8:
        st["dA_q"] = workspace_item(ws, L.cfg, which, B.MOK_ITEM_DA_Q).view(-1, 2 * I)
        st["dA_s"] = workspace_item(ws, L.cfg, which, B.MOK_ITEM_DA_SCALE).view(-1, 2 * I // 32)
    return st


def _rows_of(st, sorted_r):
    """GPU intermediates of the given sorted rows (in that order)."""
    import torch
    pr = padded_rows(sorted_r, st["offsets"], st["poff"])
    rt = torch.from_numpy(np.asarray(sorted_r, np.int64)).cuda()
    pt = torch.from_numpy(np.asarray(pr, np.int64)).cuda()
    out = dict(a=preact_rows(host(st["pre"][rt])), da=host(st["dA"][pt]),
               sh=host(st["sh"][pt]))
    if "dA_q" in st:
        out["da_q"] = st["dA_q"][pt].cpu().numpy()
        out["da_s"] = st["dA_s"][pt].cpu().numpy()
        out["daq"] = oracle.mxfp8_dequantize(out["da_q"], out["da_s"])
    return out


def check_tokens(g, st, x, w13, w2, dy, mx, tokens, mxw=None, tag=""):
    """Token-local outputs (dx, d_topk_w, d_logits) and the per-row intermediates of the
    sampled tokens' routed rows."""
    T, K, E = g["T"], g["K"], g["E"]
    idx, w = g["idx"], g["w"]
    mode = oracle.MXFP8 if mx else oracle.BF16
    tol = TOL_MXFP8 if mx else TOL_BF16
    used, idx_r = remap_experts(idx[tokens])
    xs = oracle.bf16_to_f64(x[tokens])
    dys = oracle.bf16_to_f64(dy[tokens])
    ws13, ws2 = w13[used], w2[used]
    sub_mxw = None
    if mx:
        sub_mxw = tuple((q[used], s[used]) for q, s in mxw) if mxw is not None else None
    run = lambda **kw: oracle.backward(xs, idx_r, w[tokens], ws13, ws2, dys,  # noqa: E731
                                       weight_grads=False, mode=mode, store=oracle.STORE_BF16,
                                       mx_weights=sub_mxw, **kw)
    gr = _rows_of(st, sorted_rows(st["inv"], tokens, K))
    # A
    dx_o, _, _, dtk_o, sdx, _, _, ro = run(with_slack=True, rows=("a", "a_slack",
                                                                  "dtopk_slack"))
    sdtk = ro["dtopk_slack"].reshape(dtk_o.shape)
    check_exact("bwd A" + tag, gr["a"], ro["a"], ro["a_slack"])
    # dA, w*h, dA codes, d_topk_w from the GPU's A
    names = ("da", "da_slack", "sh", "sh_slack") + (("da_q", "da_scale", "daq_slack")
                                                    if mx else ())
    _, _, _, dtk_a, ra = run(rows=names, given={"a_in": gr["a"]})
    check_exact("bwd dA | gpu A" + tag, gr["da"], ra["da"], ra["da_slack"])
    check_exact("bwd w*h | gpu A" + tag, gr["sh"], ra["sh"], ra["sh_slack"])
    if mx:
        check_codes("bwd dA codes | gpu A" + tag, gr["da_q"], gr["da_s"], ra["da_q"],
                    ra["da_scale"], ra["daq_slack"])
    dtk_g = host(g["dtk"])[tokens]
    # dS = <G, h> is an fp32 sum of fp32 products: no rounding decision, fp32 error only
    check_tol("bwd d_topk_w | gpu A" + tag, dtk_g, dtk_a, None, 2e-3)
    dlg_g = host(g["dlg"])[tokens]
    check_tol("bwd d_logits | gpu d_topk_w" + tag, dlg_g,
              oracle.router_grad(idx[tokens], w[tokens], dtk_g, E), None, 1e-5)
    # dx from the GPU's dA (MXFP8: its dequantized dA codes)
    given = {"a_in": gr["a"], "da_in": gr["da"], "sh_in": gr["sh"]}
    if mx:
        given["daq_in"] = gr["daq"]
    dx_s, _, _, _, sdx_s, _, _ = run(with_slack=True, given=given)
    dx_g = host(g["dx"])[tokens]
    check_exact("bwd dx | gpu dA" + tag, dx_g, dx_s, sdx_s, max_flagged=0.35)
    # end to end
    check_tol("bwd dx e2e" + tag, dx_g, dx_o, sdx, tol, max_slack_rms=1.2 if mx else 0.4)
    check_tol("bwd d_topk_w e2e" + tag, dtk_g, dtk_o, sdtk, tol)
    check_tol("bwd d_logits e2e" + tag, dlg_g,
              oracle.router_grad(idx[tokens], w[tokens], dtk_o, E),
              oracle.router_grad_slack(idx[tokens], w[tokens], sdtk, E), tol)


def check_expert(g, st, x, w13, w2, dy, mx, e, mxw=None, tag=""):
    """dW13[e], dW2[e]: from the GPU's own dA and w*h (bit-exact except flagged roundings),
    and end to end."""
    K = g["K"]
    idx, w = g["idx"], g["w"]
    mode = oracle.MXFP8 if mx else oracle.BF16
    tol = TOL_MXFP8 if mx else TOL_BF16
    r0, r1 = int(st["offsets"][e]), int(st["offsets"][e + 1])
    f = st["perm"][r0:r1]                       # ascending flat ids of expert e's rows
    t_e, k_e = f // K, f % K
    xe = oracle.bf16_to_f64(x[t_e])
    dye = oracle.bf16_to_f64(dy[t_e])
    sub_mxw = tuple((q[[e]], s[[e]]) for q, s in mxw) if (mx and mxw is not None) else None
    run = lambda **kw: oracle.backward(xe, np.zeros((len(f), 1), np.int32),  # noqa: E731
                                       w[t_e, k_e][:, None], w13[[e]], w2[[e]], dye,
                                       mode=mode, store=oracle.STORE_BF16, with_slack=True,
                                       mx_weights=sub_mxw, **kw)
    g13, g2 = host(g["dw13"][e]), host(g["dw2"][e])
    if len(f) == 0:
        assert np.all(g13 == 0) and np.all(g2 == 0)
        return
    gr = _rows_of(st, np.arange(r0, r1))
    _, d13, d2, _, _, s13, s2 = run(given={"a_in": gr["a"], "da_in": gr["da"],
                                           "sh_in": gr["sh"]})
    check_exact("bwd dW13 | gpu dA" + tag, g13, d13[0], s13[0], max_flagged=0.35)
    check_exact("bwd dW2 | gpu w*h" + tag, g2, d2[0], s2[0], max_flagged=0.35)
    _, d13o, d2o, _, _, s13o, s2o = run()
    check_tol("bwd dW13 e2e" + tag, g13, d13o[0], s13o[0], tol, max_slack_rms=0.6)
    check_tol("bwd dW2 e2e" + tag, g2, d2o[0], s2o[0], tol, max_slack_rms=0.6)


def check_expert_features(g, st, x, w13, w2, dy, e, feats, tag=""):
    """dW13[e] rows (gate and up) and dW2[e] columns of the features `feats` (BF16). A
    feature's weight gradients depend only on its own gate, up and W2 weights: the oracle
    runs the expert restricted to those features, a SwiGLU FFN of len(feats) features, so a
    hot expert's thousands of rows stay cheap. From the GPU's own A, dA and w*h, then end to
    end."""
    K, I = g["K"], w2.shape[2]
    idx, w = g["idx"], g["w"]
    feats = np.asarray(feats, np.int64)
    cols = np.concatenate([feats, I + feats])          # gate rows, then up rows
    r0, r1 = int(st["offsets"][e]), int(st["offsets"][e + 1])
    f = st["perm"][r0:r1]
    t_e, k_e = f // K, f % K
    g13 = host(g["dw13"][e])[cols]
    g2 = host(g["dw2"][e])[:, feats]
    if len(f) == 0:
        assert np.all(g13 == 0) and np.all(g2 == 0)
        return
    run = lambda **kw: oracle.backward(  # noqa: E731
        oracle.bf16_to_f64(x[t_e]), np.zeros((len(f), 1), np.int32), w[t_e, k_e][:, None],
        w13[[e]][:, cols], w2[[e]][:, :, feats], oracle.bf16_to_f64(dy[t_e]),
        mode=oracle.BF16, store=oracle.STORE_BF16, with_slack=True, **kw)
    gr = _rows_of(st, np.arange(r0, r1))
    _, d13, d2, _, _, s13, s2 = run(given={"a_in": gr["a"][:, cols], "da_in": gr["da"][:, cols],
                                           "sh_in": gr["sh"][:, feats]})
    # the oracle's error window of a sum over n rows grows as sqrt(n / 2048) beyond 2048 rows
    # (oracle_dot_rel_rows), and with it the share of roundings it cannot decide: at 65535
    # rows the measured fp32 error reaches about a quarter of a bf16 step
    cap = 0.35 if len(f) <= 2048 else min(0.75, 0.35 * np.sqrt(len(f) / 2048))
    check_exact("bwd dW13 | gpu dA" + tag, g13, d13[0], s13[0], max_flagged=cap)
    check_exact("bwd dW2 | gpu w*h" + tag, g2, d2[0], s2[0], max_flagged=cap)
    _, d13o, d2o, _, _, s13o, s2o = run()
    check_tol("bwd dW13 e2e" + tag, g13, d13o[0], s13o[0], TOL_BF16, max_slack_rms=0.6)
    check_tol("bwd dW2 e2e" + tag, g2, d2o[0], s2o[0], TOL_BF16, max_slack_rms=0.6)
