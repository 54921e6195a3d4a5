"""The W4A16 MoE layer on the GPU (indexed and grouped layouts) against the oracle.

Tolerance (element-wise, on bf16 values): |out - ref| <= 1e-2*|ref| +
1e-3*rms(ref).  The check is split at the bf16 rounding of the intermediate h
(see gpu_util): h against the oracle's h, then the output against the oracle's
down GEMM + combine applied to the GPU's own h.  The end-to-end ratio against
the oracle's full pipeline is printed beside it.  Sizes span several tiles and
ragged tails; the full workloads compare every row the oracle can produce in
seconds, else a sample of tokens (each token's output depends only on its own
routing, so a sub-batch of tokens run through the oracle gives those rows)."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_close_bf16, bf16_to_np, check_fp64_anchor, check_h, dev_tensor,
                      e2e_ratio, h_by_pair, weights_to)
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def chord():
    import w4a16_int4_mixture_gb300 as m
    m.build()
    return m


class Run:
    """GPU outputs of one indexed layer call plus its routing layout."""

    def __init__(self, out, h, si, ei, ntp, bm):
        self.out, self.h, self.si, self.ei, self.ntp, self.bm = out, h, si, ei, ntp, bm


def run_indexed_full(chord, inp, block_m=None, flags=0, weights=None):
    s = inp.shape
    bm = block_m or s.block_m
    w = weights or weights_to(inp, DEV)
    x = dev_tensor(inp.x, DEV, True)
    ids = dev_tensor(inp.topk_ids, DEV)
    tw = dev_tensor(inp.topk_weights, DEV)
    emap = None if inp.expert_map is None else dev_tensor(inp.expert_map, DEV)
    si, ei, ntp = chord.moe_align(ids, s.E_global, s.E_local, bm, expert_map=emap)
    h = torch.empty((si.numel(), s.I), dtype=torch.bfloat16, device=DEV)
    out = chord.w4a16_moe_indexed(x, *w, tw, si, ei, ntp, bm, s.E_global, flags=flags | 1,
                                  h_out=h)
    torch.cuda.synchronize()
    return Run(bf16_to_np(out), bf16_to_np(h), si.cpu().numpy(), ei.cpu().numpy(),
               int(ntp.item()), bm)


def run_indexed(chord, inp, block_m=None, flags=0, weights=None):
    return run_indexed_full(chord, inp, block_m, flags, weights).out


def sub_batch(inp, tokens):
    s = inp.shape
    sub = synth.MoEShape(s.name + "-sub", T=len(tokens), k=s.k, E_global=s.E_global,
                         E_local=s.E_local, H=s.H, I=s.I, block_m=s.block_m, seed=s.seed)
    return synth.MoEInputs(sub, inp.x[tokens], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                           inp.topk_ids[tokens], inp.topk_weights[tokens], inp.expert_map)


def verify_indexed(inp, run, tokens=None, label=""):
    """Split check of an indexed layer run (see gpu_util): rows of `tokens`
    (all tokens when None) against the oracle on the same tokens, and both
    against the fp64 evaluation of the definition (gpu_util.check_fp64_anchor).
    Returns the end-to-end ratio against the oracle (reported, not asserted)."""
    s = inp.shape
    if tokens is None:
        tokens = np.arange(s.T)
    sub = sub_batch(inp, tokens)
    (rsi, rei, rntp), (ref_out, ref_h, _) = oracle.run_workload(sub, block_m=run.bm, want_h=True)
    # GPU rows of the sub-batch's pairs, in the oracle's row order
    pos = np.full(s.T * s.k, -1, np.int64)
    body = run.si[:run.ntp]
    real = body < s.T * s.k
    pos[body[real]] = np.nonzero(real)[0]
    h_sub = np.zeros_like(ref_h)
    valid = np.zeros(rsi.size, bool)
    for r in range(rntp):
        p_sub = rsi[r]
        if p_sub >= sub.shape.T * s.k:
            continue
        t_sub, j = divmod(int(p_sub), s.k)
        r_gpu = pos[int(tokens[t_sub]) * s.k + j]
        assert r_gpu >= 0, "pair missing from the GPU layout"
        h_sub[r] = run.h[r_gpu]
        valid[r] = True
    flips = check_h(h_sub[valid], ref_h[valid], f"{label} h")
    down_ref = oracle.moe_indexed_down(h_sub, inp.w2_q, inp.w2_s, sub.topk_weights, rsi, rei,
                                       rntp, run.bm, sub.shape.T, s.k)
    got = run.out[tokens]
    assert_close_bf16(got, down_ref, f"{label} output given h")
    ratio = e2e_ratio(got, ref_out)
    fg, fo, rg, ro = check_fp64_anchor(
        inp, tokens, h_by_pair(h_sub[valid], rsi[valid], s.k, tokens),
        got, h_by_pair(ref_h[valid], rsi[valid], s.k, tokens), ref_out,
        f"{label} against fp64")
    print(f"[{label}] h flips vs oracle {100 * flips:.4f}%  end-to-end worst {ratio:.3f}x | "
          f"vs fp64: h flips gpu {100 * fg:.3f}% oracle {100 * fo:.3f}%, worst gpu {rg:.2f}x "
          f"oracle {ro:.2f}x")
    return ratio


def small(T, k, Eg, El, H, I, seed, bm=16, emap=True, sigma=0.05):
    s = synth.MoEShape("small", T=T, k=k, E_global=Eg, E_local=El, H=H, I=I, block_m=bm, seed=seed)
    inp = synth.make_inputs(s)
    rng = np.random.default_rng(seed + 100)
    if El < Eg and emap:
        m = np.full(Eg, -1, np.int32)
        m[rng.permutation(Eg)[:El]] = np.arange(El, dtype=np.int32)
        inp.expert_map = m
    inp.w13_s = synth.scales(rng, El, 2 * I, H, sigma=sigma)
    inp.w2_s = synth.scales(rng, El, H, I, sigma=sigma)
    return inp


SMALL = {
    "tiny": lambda: synth.make_inputs(synth.workload("tiny")),
    "decode32-map": lambda: small(40, 3, 10, 6, 512, 256, 1),
    "decode64": lambda: small(64, 4, 8, 8, 512, 256, 2, emap=False),
    "decode128": lambda: small(100, 4, 8, 8, 256, 128, 3, emap=False),
    "prefill": lambda: small(300, 2, 3, 3, 256, 128, 4, emap=False),
    "prefill-multichunk": lambda: small(700, 2, 3, 3, 256, 256, 5, emap=False),
    "single-token": lambda: small(1, 8, 16, 16, 256, 128, 6, emap=False),
    "topk1": lambda: small(50, 1, 4, 4, 768, 384, 7, emap=False),
    "many-units-long-k": lambda: small(320, 4, 16, 16, 2048, 512, 8, emap=False),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_indexed_small(chord, name):
    inp = SMALL[name]()
    verify_indexed(inp, run_indexed_full(chord, inp), label=name)


@pytest.mark.parametrize("bm", [1, 8, 32, 64])
def test_indexed_block_m(chord, bm):
    inp = small(40, 3, 10, 6, 512, 256, 11)
    verify_indexed(inp, run_indexed_full(chord, inp, block_m=bm), label=f"block_m={bm}")


def test_indexed_deterministic_path(chord):
    inp = small(60, 4, 12, 8, 512, 256, 12)
    a = run_indexed_full(chord, inp, flags=2)
    b = run_indexed_full(chord, inp, flags=2)
    verify_indexed(inp, a, label="deterministic combine")
    assert np.array_equal(a.out, b.out), "deterministic path is not bit-reproducible"
    assert np.array_equal(a.h, b.h)


def test_tokens_without_local_experts_are_zero(chord):
    inp = small(30, 2, 8, 4, 256, 128, 13)
    nonlocal_ids = np.nonzero(inp.expert_map < 0)[0]
    inp.topk_ids[:5] = nonlocal_ids[:2]
    run = run_indexed_full(chord, inp)
    assert np.all(run.out[:5] == 0)
    verify_indexed(inp, run, label="no-local tokens")


def test_zero_weights_give_zero(chord):
    inp = small(20, 2, 4, 4, 256, 128, 14, emap=False)
    inp.w13_q[:] = np.int32(np.uint32(0x88888888).view(np.int32))
    got = run_indexed(chord, inp)
    assert np.all(oracle.bf16_to_f32(got) == 0)


def test_poisoned_workspace_does_not_leak(chord):
    """Stale NaN bytes in the workspace and h buffer must not reach the output."""
    inp = small(40, 3, 10, 6, 512, 256, 15)
    s = inp.shape
    ws = torch.full((64 << 20,), 0xFF, dtype=torch.uint8, device=DEV)  # NaN patterns
    w = weights_to(inp, DEV)
    x = dev_tensor(inp.x, DEV, True)
    si, ei, ntp = chord.moe_align(dev_tensor(inp.topk_ids, DEV), s.E_global, s.E_local, 16,
                                  expert_map=dev_tensor(inp.expert_map, DEV))
    for flags in (0, 2):
        h = torch.full((si.numel(), s.I), float("nan"), dtype=torch.bfloat16, device=DEV)
        out = chord.w4a16_moe_indexed(x, *w, dev_tensor(inp.topk_weights, DEV), si, ei, ntp, 16,
                                      s.E_global, workspace=ws, flags=flags | 1, h_out=h)
        torch.cuda.synchronize()
        run = Run(bf16_to_np(out), bf16_to_np(h), si.cpu().numpy(), ei.cpu().numpy(),
                  int(ntp.item()), 16)
        verify_indexed(inp, run, label=f"poisoned workspace flags={flags}")
        # h rows of the layout's sentinel (padding) entries are zero
        pad = np.nonzero(run.si[:run.ntp] >= s.T * s.k)[0]
        assert pad.size > 0 and np.all(run.h[pad] == 0), "sentinel rows of h are not zero"


# ---------------------------------------------------------------- grouped
def contiguous_layer_check(chord, inp, align, label, flags=0, weights=None):
    s = inp.shape
    a2, m_idx, r2p = synth.grouped_contiguous_layout(inp, align=align)
    w = weights or weights_to(inp, DEV)
    h = torch.empty((a2.shape[0], s.I), dtype=torch.bfloat16, device=DEV)
    rows, toks = chord.w4a16_moe_grouped("contiguous", dev_tensor(a2, DEV, True), *w,
                                         m_indices=dev_tensor(m_idx, DEV),
                                         row_to_pair=dev_tensor(r2p, DEV),
                                         topk_weights=dev_tensor(inp.topk_weights, DEV),
                                         flags=flags | 1, h_out=h)
    torch.cuda.synchronize()
    ref_rows, ref_tok, ref_h = oracle.moe_grouped("contiguous", a2, inp.w13_q, inp.w13_s,
                                                  inp.w2_q, inp.w2_s, m_indices=m_idx,
                                                  row_to_pair=r2p, topk_weights=inp.topk_weights,
                                                  T=s.T, k=s.k, want_h=True)
    valid = m_idx >= 0
    hg = bf16_to_np(h)
    hg[~valid] = 0
    check_h(hg[valid], ref_h[valid], f"{label} h")
    d_rows, d_tok = oracle.moe_grouped_down("contiguous", hg, inp.w2_q, inp.w2_s,
                                            m_indices=m_idx, row_to_pair=r2p,
                                            topk_weights=inp.topk_weights, T=s.T, k=s.k)
    assert_close_bf16(bf16_to_np(rows)[valid], d_rows[valid], f"{label} rows given h")
    assert_close_bf16(bf16_to_np(toks), d_tok, f"{label} tokens given h")
    fg, fo, rg, ro = check_fp64_anchor(inp, np.arange(s.T), h_by_pair(hg, r2p, s.k),
                                       bf16_to_np(toks), h_by_pair(ref_h, r2p, s.k), ref_tok,
                                       f"{label} against fp64")
    print(f"[{label}] end-to-end tokens {e2e_ratio(bf16_to_np(toks), ref_tok):.3f}x | vs fp64: "
          f"h flips gpu {100 * fg:.3f}% oracle {100 * fo:.3f}%, worst gpu {rg:.2f}x oracle "
          f"{ro:.2f}x")
    return bf16_to_np(rows)[valid], bf16_to_np(toks)


@pytest.mark.parametrize("align", [16, 128])
def test_grouped_contiguous(chord, align):
    contiguous_layer_check(chord, small(80, 3, 10, 6, 512, 256, 21), align,
                           f"contiguous align={align}")


def masked_layer_check(chord, inp, a3, mm, r2p, w, label):
    s = inp.shape
    exp_m = int(np.ceil(mm.sum() / s.E_local))
    M = a3.shape[0] * a3.shape[1]
    h = torch.empty((M, s.I), dtype=torch.bfloat16, device=DEV)
    rows, toks = chord.w4a16_moe_grouped("masked", dev_tensor(a3, DEV, True), *w,
                                         masked_m=dev_tensor(mm, DEV), expected_m=exp_m,
                                         row_to_pair=dev_tensor(r2p, DEV),
                                         topk_weights=dev_tensor(inp.topk_weights, DEV), flags=1,
                                         h_out=h)
    torch.cuda.synchronize()
    ref_rows, ref_tok, ref_h = oracle.moe_grouped("masked", a3, inp.w13_q, inp.w13_s, inp.w2_q,
                                                  inp.w2_s, masked_m=mm, row_to_pair=r2p,
                                                  topk_weights=inp.topk_weights, T=s.T, k=s.k,
                                                  want_h=True)
    valid = r2p >= 0
    hg = bf16_to_np(h)
    hg[~valid] = 0
    flips = check_h(hg[valid], ref_h[valid], f"{label} h")
    d_rows, d_tok = oracle.moe_grouped_down("masked", hg, inp.w2_q, inp.w2_s, masked_m=mm,
                                            max_m=a3.shape[1], row_to_pair=r2p,
                                            topk_weights=inp.topk_weights, T=s.T, k=s.k)
    assert_close_bf16(bf16_to_np(rows)[valid], d_rows[valid], f"{label} rows given h")
    assert_close_bf16(bf16_to_np(toks), d_tok, f"{label} tokens given h")
    fg, fo, rg, ro = check_fp64_anchor(inp, np.arange(s.T), h_by_pair(hg, r2p, s.k),
                                       bf16_to_np(toks), h_by_pair(ref_h, r2p, s.k), ref_tok,
                                       f"{label} against fp64")
    print(f"[{label}] h flips {100 * flips:.4f}%  end-to-end tokens "
          f"{e2e_ratio(bf16_to_np(toks), ref_tok):.3f}x | vs fp64: h flips gpu {100 * fg:.3f}% "
          f"oracle {100 * fo:.3f}%, worst gpu {rg:.2f}x oracle {ro:.2f}x")
    return bf16_to_np(toks)


def test_grouped_masked(chord):
    inp = small(80, 3, 10, 6, 512, 256, 22)
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    masked_layer_check(chord, inp, a3, mm, r2p, weights_to(inp, DEV), "masked")


def test_grouped_matches_indexed(chord):
    """Same draw through both entry points."""
    inp = small(64, 4, 8, 8, 512, 256, 23, emap=False)
    ind = run_indexed_full(chord, inp)
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    toks = masked_layer_check(chord, inp, a3, mm, r2p, weights_to(inp, DEV), "masked-vs-indexed")
    assert_close_bf16(toks, ind.out, "grouped vs indexed tokens")


# ---------------------------------------------------------------- CUDA graphs
def test_graph_capture_token_sweep(chord):
    """One weight set, routing buffers over-allocated for the largest T, one
    captured graph per token count; replays match eager calls bit-exactly
    (deterministic combine) and the split check."""
    Tmax, k, Eg, H, I = 256, 8, 64, 512, 256
    base = small(Tmax, k, Eg, Eg, H, I, 31, emap=False)
    w = weights_to(base, DEV)
    cap = chord.moe_align_capacity(Tmax, k, Eg, 16)
    si = torch.empty(cap, dtype=torch.int32, device=DEV)
    ei = torch.empty(cap // 16, dtype=torch.int32, device=DEV)
    ntp = torch.empty(1, dtype=torch.int32, device=DEV)
    x_all = dev_tensor(base.x, DEV, True)
    ids_all = dev_tensor(base.topk_ids, DEV)
    tw_all = dev_tensor(base.topk_weights, DEV)
    for T in (1, 16, 128, 256):
        x, ids, tw = x_all[:T].contiguous(), ids_all[:T].contiguous(), tw_all[:T].contiguous()
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        ws_a = torch.empty(chord.ops.align_workspace_size(Tmax, k, Eg), dtype=torch.uint8,
                           device=DEV)
        ws_l = torch.empty(chord.moe_workspace_size(T, k, Eg, Eg, H, I, 16, cap, 2),
                           dtype=torch.uint8, device=DEV)
        h = torch.empty((cap, I), dtype=torch.bfloat16, device=DEV)

        def step():
            chord.moe_align(ids, Eg, Eg, 16, capacity=cap, workspace=ws_a, out=(si, ei, ntp))
            chord.w4a16_moe_indexed(x, *w, tw, si, ei, ntp, 16, Eg, out=out, workspace=ws_l,
                                    h_out=h, flags=2)

        step()
        torch.cuda.synchronize()
        eager = bf16_to_np(out).copy()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step()
        torch.cuda.current_stream().wait_stream(s)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        replay = bf16_to_np(out)
        assert np.array_equal(replay, eager), f"graph replay differs from eager T={T}"
        sub = sub_batch(base, np.arange(T))
        run = Run(replay, bf16_to_np(h), si.cpu().numpy(), ei.cpu().numpy(), int(ntp.item()), 16)
        verify_indexed(sub, run, label=f"graph T={T}")


def test_tp8_graph_capture_over_allocated(chord):
    """The TP8 configuration as a server runs it: one packed weight set (384
    experts, hidden 7168, intermediate 256), one set of routing buffers and one
    workspace sized once for 2048 tokens, and one CUDA graph captured per token
    count T in {1, 16, 128, 2048} on those same buffers (page: "vLLM
    integration": over-allocated moe_align buffers consumed without host
    readback).  Each replay equals the eager call bit for bit (ordered
    combine) and is checked against the oracle and the fp64 evaluation
    (sampled tokens at 2048)."""
    Tmax = 2048
    base = synth.make_inputs(synth.workload("tp8", T=Tmax))
    s0 = base.shape
    pw = chord.prepack_weights(*weights_to(base, DEV))
    w = (pw, None, None, None)
    cap = chord.moe_align_capacity(Tmax, s0.k, s0.E_local, 16)
    si = torch.empty(cap, dtype=torch.int32, device=DEV)
    ei = torch.empty(cap // 16, dtype=torch.int32, device=DEV)
    ntp = torch.empty(1, dtype=torch.int32, device=DEV)
    h = torch.empty((cap, s0.I), dtype=torch.bfloat16, device=DEV)
    out_all = torch.empty((Tmax, s0.H), dtype=torch.bfloat16, device=DEV)
    ws_a = torch.empty(chord.ops.align_workspace_size(Tmax, s0.k, s0.E_local), dtype=torch.uint8,
                       device=DEV)
    ws_l = torch.empty(chord.moe_workspace_size(Tmax, s0.k, s0.E_global, s0.E_local, s0.H, s0.I,
                                                16, cap, 2), dtype=torch.uint8, device=DEV)
    x_all = dev_tensor(base.x, DEV, True)
    ids_all = dev_tensor(base.topk_ids, DEV)
    tw_all = dev_tensor(base.topk_weights, DEV)
    for T in (1, 16, 128, 2048):
        x, ids, tw, out = x_all[:T], ids_all[:T], tw_all[:T], out_all[:T]
        assert chord.moe_workspace_size(T, s0.k, s0.E_global, s0.E_local, s0.H, s0.I, 16, cap,
                                        2) <= ws_l.numel()

        def step():
            chord.moe_align(ids, s0.E_global, s0.E_local, 16, capacity=cap, workspace=ws_a,
                            out=(si, ei, ntp))
            chord.w4a16_moe_indexed(x, *w, tw, si, ei, ntp, 16, s0.E_global, out=out,
                                    workspace=ws_l, h_out=h, flags=2)

        step()
        torch.cuda.synchronize()
        eager = bf16_to_np(out).copy()
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            with torch.cuda.graph(g, stream=st):
                step()
        torch.cuda.current_stream().wait_stream(st)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        replay = bf16_to_np(out)
        assert np.array_equal(replay, eager), f"graph replay differs from eager T={T}"
        sub = sub_batch(base, np.arange(T))
        run = Run(replay, bf16_to_np(h), si.cpu().numpy(), ei.cpu().numpy(), int(ntp.item()), 16)
        tokens = None if T <= 128 else np.random.default_rng(9).choice(T, 48, replace=False)
        verify_indexed(sub, run, tokens, label=f"TP8 graph T={T}, buffers for {Tmax}")
        del g


# ---------------------------------------------------------------- full workloads
@pytest.fixture(scope="module")
def ep8_weights():
    s = synth.workload("ep8-decode")
    inp = synth.make_inputs(s)
    return inp, weights_to(inp, DEV)


def _with_weights(inp_w, wl, T=None):
    base, w = inp_w
    s = synth.workload(wl, T=T)
    r = synth.make_inputs(s, weights=False)
    r.w13_q, r.w13_s, r.w2_q, r.w2_s = base.w13_q, base.w13_s, base.w2_q, base.w2_s
    return r, w


def test_ep8_decode_full(chord, ep8_weights):
    inp, w = _with_weights(ep8_weights, "ep8-decode")
    verify_indexed(inp, run_indexed_full(chord, inp, weights=w), label="EP8 decode T=512")


def test_ep8_decode_deterministic(chord, ep8_weights):
    inp, w = _with_weights(ep8_weights, "ep8-decode")
    a = run_indexed_full(chord, inp, weights=w, flags=2)
    b = run_indexed_full(chord, inp, weights=w, flags=2)
    assert np.array_equal(a.out, b.out)
    tokens = np.random.default_rng(2).choice(inp.shape.T, 64, replace=False)
    verify_indexed(inp, a, tokens, label="EP8 decode T=512 ordered combine")


def test_ep8_prefill_sampled(chord, ep8_weights):
    inp, w = _with_weights(ep8_weights, "ep8-prefill")
    run = run_indexed_full(chord, inp, weights=w)
    assert np.all(np.isfinite(oracle.bf16_to_f32(run.out)))
    tokens = np.random.default_rng(0).choice(inp.shape.T, 48, replace=False)
    verify_indexed(inp, run, tokens, label="EP8 prefill T=8192 (48 sampled tokens)")


def test_skewed_indexed_and_masked(chord, ep8_weights):
    inp, w = _with_weights(ep8_weights, "skewed")
    verify_indexed(inp, run_indexed_full(chord, inp, weights=w), label="Zipf indexed")
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    masked_layer_check(chord, inp, a3, mm, r2p, w, "Zipf masked")


@pytest.mark.parametrize("T", [1, 16, 128, 2048])
def test_tp8(chord, T):
    s = synth.workload("tp8", T=T)
    inp = synth.make_inputs(s)
    run = run_indexed_full(chord, inp)
    tokens = None if T <= 128 else np.random.default_rng(1).choice(T, 64, replace=False)
    verify_indexed(inp, run, tokens, label=f"TP8 T={T}")


@pytest.mark.parametrize("shape", ["prefill-multiunit", "decode-multiunit"])
def test_gate_up_bit_reproducible(chord, shape):
    """The gate/up output is computed without atomics, so repeated runs must be
    bit-identical.  Run many times on shapes where every CTA walks several work
    units: this catches shared-memory / tensor-memory races between the roles
    (it caught a missing async-proxy fence before a codes stage was reused)."""
    if shape == "prefill-multiunit":
        inp = small(2048, 8, 48, 48, 1024, 512, 40, emap=False)
    else:
        inp = small(512, 8, 64, 64, 2048, 1024, 41, emap=False)
    s = inp.shape
    w = weights_to(inp, DEV)
    x = dev_tensor(inp.x, DEV, True)
    si, ei, ntp = chord.moe_align(dev_tensor(inp.topk_ids, DEV), s.E_global, s.E_local, 16)
    tw = dev_tensor(inp.topk_weights, DEV)
    ref = None
    for _ in range(12):
        h = torch.full((si.numel(), s.I), float("nan"), dtype=torch.bfloat16, device=DEV)
        chord.w4a16_moe_indexed(x, *w, tw, si, ei, ntp, 16, s.E_global, flags=1, h_out=h)
        torch.cuda.synchronize()
        cur = h[:int(ntp.item())].view(torch.int16).cpu()
        if ref is None:
            ref = cur
        else:
            assert torch.equal(cur, ref), "gate/up output changed between identical runs"
