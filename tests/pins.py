"""Pins of the CPU oracle: checks against what the Chord W4A16 MoE page and
plain mathematics fix, written independently of oracle.c.

Each pin returns (ok: bool, detail: str) so that the same checks serve both the
plain pin tests and the planted-mistake tests (a pin must fail when one mistake
is planted in the oracle).

Independent pieces used here (none calls oracle.c):
  * rne_bf16: round-to-nearest-even to bf16 of float64 values through
    frexp / rint (not the bit trick oracle.c uses);
  * decode_codes: nibble extraction with numpy shifts;
  * brute_force_token: a per-token fp64 evaluation of the expert MLP and the
    combine, one token at a time.
"""

from __future__ import annotations

import numpy as np

import oracle
from w4a16_int4_mixture_gb300 import synth

BF16_MAX = float.fromhex("0x1.fep127")


def rne_bf16(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.  Handles
    normal, subnormal, overflow (to inf), inf and NaN."""
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    fin = np.isfinite(v)
    out[~fin] = v[~fin]
    x = v[fin]
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    # bf16 keeps 8 significant bits for normals; below 2**-126 the spacing is 2**-133
    e_eff = np.maximum(e, -125)
    q = np.rint(np.ldexp(x, 8 - e_eff))     # rint rounds half to even
    r = np.ldexp(q, e_eff - 8)
    # values at or beyond max + half an ulp round to infinity
    limit = BF16_MAX + float.fromhex("0x1p119")
    r = np.where(np.abs(x) >= limit, np.copysign(np.inf, x), r)
    out[fin] = r
    return out


def f64_to_bf16_bits(v) -> np.ndarray:
    """Bits of float64 values that are already bf16 values (exact narrowing)."""
    v = np.asarray(v, dtype=np.float64)
    b = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return b


def bf16_bits_to_f64(b) -> np.ndarray:
    return oracle.bf16_to_f32(np.asarray(b, dtype=np.uint16)).astype(np.float64)


def decode_codes(wq: np.ndarray) -> np.ndarray:
    """[..., K/8] int32 words -> [..., K] codes, element 8w+i from bits [4i, 4i+4)."""
    w = np.asarray(wq).view(np.uint32)
    sh = (np.arange(8, dtype=np.uint32) * 4)
    c = (w[..., None] >> sh) & np.uint32(0xF)
    return c.reshape(w.shape[:-1] + (w.shape[-1] * 8,)).astype(np.int64)


def dequant_f64(wq: np.ndarray, ws: np.ndarray) -> np.ndarray:
    """Reference dequant of one [N, K] weight, float64 holding bf16 values."""
    q = decode_codes(wq)
    K = q.shape[-1]
    s = bf16_bits_to_f64(ws)
    s_full = np.repeat(s, 32, axis=-1)[..., :K]
    return rne_bf16((q - 8).astype(np.float64) * s_full)


# FP4 E2M1 values of codes 0..7 as the OCP Microscaling formats list them;
# codes 8..15 are the same magnitudes with the sign bit set
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def dequant_mx_f64(wq: np.ndarray, ws8: np.ndarray) -> np.ndarray:
    """Reference MXFP4 dequant of one [N, K] weight: E2M1 code values from the
    table above times 2^(s - 127) per 32 channels, float64 (exact for finite
    values; bf16 rounding only changes values that overflow it)."""
    q = decode_codes(wq)
    mag = np.array(E2M1_VALUES)[q & 7]
    v = np.where(q >= 8, -mag, mag)
    K = q.shape[-1]
    sc = np.repeat(ws8.astype(np.int64), 32, axis=-1)[..., :K]
    return rne_bf16(np.ldexp(v, sc - 127))


def silu64(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def rounding_ratio(got, ref) -> float:
    """max |got - ref| / (ulp_bf16(ref)/2 + 1e-4 * rms(ref)): got is ref rounded
    to bf16 up to fp32 accumulation error when this is <= 1."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    ulp_r = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 1e-30))[1] - 8)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref) / (0.5 * ulp_r + 1e-4 * rms + 1e-30)))


def tolerance_violation(out, ref) -> float:
    """max over elements of |out-ref| / (1e-2*|ref| + 1e-3*rms(ref)); <= 1 passes."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = 1e-2 * np.abs(ref) + 1e-3 * rms
    err = np.abs(out - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    return float(np.max(ratio))


# --------------------------------------------------------------------------
# brute force: one token at a time, fp64, straight from the definition
# --------------------------------------------------------------------------
def brute_force_token(inp: synth.MoEInputs, t: int, local_of_slot, deq=None):
    """fp64 output row of token t: sum over local slots j of
    w[t,j] * W2_e (bf16(silu(W13_e[:I] x) * (W13_e[I:] x))).  Also returns the
    per-slot pre-rounding (g, u) for finer checks."""
    s = inp.shape
    x = bf16_bits_to_f64(inp.x[t])
    acc = np.zeros(s.H, dtype=np.float64)
    parts = []
    for j in range(s.k):
        e = local_of_slot[t, j]
        if e < 0:
            continue
        W13 = (deq or dequant_f64)(inp.w13_q[e], inp.w13_s[e])
        W2 = (deq or dequant_f64)(inp.w2_q[e], inp.w2_s[e])
        g = W13[:s.I] @ x
        u = W13[s.I:] @ x
        h = rne_bf16(silu64(g) * u)
        y = W2 @ h
        acc += float(inp.topk_weights[t, j]) * y
        parts.append((j, e, g, u, h, y))
    return acc, parts


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------
def pin_dequant_exhaustive():
    """All 16 codes x all 65536 bf16 scale bit patterns vs exact RNE."""
    N, K = 65536, 32
    codes = np.tile(np.arange(32) % 16, (N, 1))
    wq = synth.pack_codes(codes)
    ws = np.arange(N, dtype=np.uint32).astype(np.uint16).reshape(N, 1)
    got = oracle.dequant(wq, ws, N, K)
    s = bf16_bits_to_f64(ws)                          # [N, 1]
    with np.errstate(invalid="ignore"):
        exact = (codes - 8).astype(np.float64) * s     # exact in float64
    want = rne_bf16(exact)
    g = got.astype(np.float64)
    both_nan = np.isnan(g) & np.isnan(want)
    same = both_nan | (f64_to_bf16_bits(np.where(np.isnan(g), 0, g)) ==
                       f64_to_bf16_bits(np.where(np.isnan(want), 0, want)))
    same &= (np.isnan(g) == np.isnan(want))
    bad = np.size(same) - int(np.count_nonzero(same))
    return bad == 0, f"{bad} mismatching dequant values"


def pin_dequant_zero_code():
    """Code 8 dequantises to exactly 0 for every finite scale."""
    N, K = 1024, 32
    wq = synth.pack_codes(np.full((N, K), 8))
    rng = np.random.default_rng(5)
    ws = (rng.integers(0, 0x7F80, size=(N, 1)) | (rng.integers(0, 2, size=(N, 1)) << 15)
          ).astype(np.uint16)
    got = oracle.dequant(wq, ws, N, K)
    return bool(np.all(got == 0.0)), "code 8 must give 0"


def pin_one_hot_structure(seed=11):
    """x = unit vector at channel c0: gate/up outputs equal one dequantised weight
    column, so nibble order, scale group axis, zero point and gate/up order are
    all visible.  Explicit codes -> packed with the storage convention."""
    rng = np.random.default_rng(seed)
    E, H, I = 2, 64, 32
    c13 = rng.integers(0, 16, size=(E, 2 * I, H))
    c2 = rng.integers(0, 16, size=(E, H, I))
    s13 = synth.scales(rng, E, 2 * I, H, sigma=0.5)
    s2 = synth.scales(rng, E, H, I, sigma=0.5)
    w13 = synth.pack_codes(c13)
    w2 = synth.pack_codes(c2)
    ok = True
    detail = ""
    for e in range(E):
        for c0 in (0, 5, 31, 32, 45, 63):
            x = np.zeros((1, H), np.uint16)
            x[0, c0] = 0x3F80  # 1.0
            g, u, h, y = oracle.expert_mlp(w13, s13, w2, s2, e, x)
            sg = bf16_bits_to_f64(s13[e, :, c0 // 32])
            col = rne_bf16((c13[e, :, c0] - 8) * sg)
            if not (np.array_equal(g[0].astype(np.float64), col[:I]) and
                    np.array_equal(u[0].astype(np.float64), col[I:])):
                ok = False
                detail = f"gate/up column mismatch e={e} c0={c0}"
    return ok, detail


def pin_down_one_hot(seed=12):
    """Down GEMM on a unit intermediate vector equals one column of W2.
    Built through the MLP with gate = +1 weights on one channel: choose codes so
    h is a known one-hot bf16 vector."""
    E, H, I = 1, 64, 32
    rng = np.random.default_rng(seed)
    # gate rows: code 9 (w=+s) on channel 0 only, else 8 (w=0); up rows likewise
    c13 = np.full((E, 2 * I, H), 8)
    i0 = 7
    c13[0, i0, 0] = 9        # gate_i0 = x0
    c13[0, I + i0, 0] = 9    # up_i0 = x0
    s13 = synth.const_scales(E, 2 * I, H, 0x3F80)
    c2 = rng.integers(0, 16, size=(E, H, I))
    s2 = synth.scales(rng, E, H, I, sigma=0.5)
    w13 = synth.pack_codes(c13)
    w2 = synth.pack_codes(c2)
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x4000  # 2.0
    g, u, h, y = oracle.expert_mlp(w13, s13, w2, s2, 0, x)
    hv = rne_bf16(silu64(2.0) * 2.0)
    h_want = np.zeros(I)
    h_want[i0] = hv
    if not np.array_equal(bf16_bits_to_f64(h[0]), h_want):
        return False, "h is not the expected one-hot vector"
    col = rne_bf16((c2[0, :, i0] - 8) * bf16_bits_to_f64(s2[0, :, i0 // 32])) * hv
    ok = np.array_equal(y[0].astype(np.float64), col)
    return ok, "down output is not the expected W2 column"


def _closed_form_inputs(code13_gate, code13_up, code2, T=6, k=3, E=4, H=64, I=32, seed=3):
    """Unit scales, small-integer activations, exact dyadic router weights."""
    rng = np.random.default_rng(seed)
    shape = synth.MoEShape("closed", T=T, k=k, E_global=E, E_local=E, H=H, I=I, block_m=4,
                           seed=seed)
    c13 = np.empty((E, 2 * I, H), np.int64)
    c13[:, :I] = code13_gate
    c13[:, I:] = code13_up
    c2 = np.full((E, H, I), code2)
    xi = rng.integers(-2, 3, size=(T, H)).astype(np.float32)
    x = (xi.view(np.uint32) >> 16).astype(np.uint16)   # small integers are bf16-exact
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = np.tile(np.array([0.5, 0.25, 0.25][:k], np.float32), (T, 1))
    inp = synth.MoEInputs(shape, x, synth.pack_codes(c13), synth.const_scales(E, 2 * I, H, 0x3F80),
                          synth.pack_codes(c2), synth.const_scales(E, H, I, 0x3F80), ids, w, None)
    return inp, xi


def pin_closed_form_equal_codes(c=11):
    """All codes c, unit scales: g = u = (c-8) * sum(x) =: G for every channel,
    h = bf16(silu(G) * G), y = (c-8) * I * h, out = y (weights sum to 1)."""
    inp, xi = _closed_form_inputs(c, c, c)
    s = inp.shape
    _, out = oracle.run_workload(inp)
    got = bf16_bits_to_f64(out)
    G = (c - 8) * xi.sum(axis=1).astype(np.float64)           # exact
    h = rne_bf16(silu64(G) * G)
    # silu in fp32 may round differently from fp64 by an ulp before the bf16
    # rounding; take the fp32 value the oracle's silu gives when they disagree
    h32 = np.array([oracle.bf16_to_f32(np.array([oracle.f32_to_bf16(
        np.float32(oracle.silu(float(v))) * np.float32(v))]))[0] for v in G], np.float64)
    y = (c - 8) * s.I * h32
    want = rne_bf16(y)[:, None] * np.ones((1, s.H))
    ok = np.array_equal(got, want) and np.max(np.abs(h - h32) / np.maximum(np.abs(h), 1e-30)) < 1e-2
    return ok, "closed form (equal codes) mismatch"


def pin_closed_form_gate_up_order():
    """Gate codes 9 (w=+1), up codes 10 (w=+2), down codes 9: with S = sum(x),
    g = S, u = 2S, h = bf16(silu(S) * 2S), y = I * h."""
    inp, xi = _closed_form_inputs(9, 10, 9)
    s = inp.shape
    _, out = oracle.run_workload(inp)
    got = bf16_bits_to_f64(out)
    S = xi.sum(axis=1).astype(np.float64)
    h = np.array([oracle.bf16_to_f32(np.array([oracle.f32_to_bf16(
        np.float32(oracle.silu(float(v))) * np.float32(2 * v))]))[0] for v in S], np.float64)
    h64 = rne_bf16(silu64(S) * 2 * S)
    y = s.I * h
    want = rne_bf16(y)[:, None] * np.ones((1, s.H))
    ok = np.array_equal(got, want) and np.allclose(h, h64, rtol=1e-2)
    return ok, "closed form (gate/up order) mismatch"


def pin_zero_weights():
    """All codes 8: every weight is 0, so the output is exactly 0."""
    inp, _ = _closed_form_inputs(8, 8, 8)
    _, out = oracle.run_workload(inp)
    return bool(np.all(bf16_bits_to_f64(out) == 0.0)), "nonzero output with zero weights"


def small_random_inputs(seed=0, T=12, k=3, Eg=6, El=5, H=64, I=32, bm=4, emap=True):
    rng = np.random.default_rng(seed)
    shape = synth.MoEShape("small", T=T, k=k, E_global=Eg, E_local=El, H=H, I=I, block_m=bm,
                           seed=seed)
    inp = synth.make_inputs(shape, seed=seed)
    # a non-identity expert map: local experts are a shuffled subset
    if emap:
        m = np.full(Eg, -1, np.int32)
        chosen = rng.permutation(Eg)[:El]
        m[chosen] = np.arange(El, dtype=np.int32)
        inp.expert_map = m
    # scales large enough that bf16 rounding of h matters
    inp.w13_s = synth.scales(rng, El, 2 * I, H, sigma=0.1)
    inp.w2_s = synth.scales(rng, El, H, I, sigma=0.1)
    return inp


def pin_brute_force(seed=0, **kw):
    """Oracle layer vs per-token fp64 brute force.  Pre-rounding g, u agree to
    fp32 accumulation error; h to one bf16 ulp; the output within a tolerance
    ten times tighter than the GPU bound."""
    inp = small_random_inputs(seed, **kw)
    s = inp.shape
    lid = synth.local_ids(inp)
    (sorted_ids, expert_ids, ntp), (out, h_rows, y_pairs) = oracle.run_workload(
        inp, want_h=True, want_y=True)
    got = bf16_bits_to_f64(out)
    ok = True
    worst = 0.0
    for t in range(s.T):
        ref, parts = brute_force_token(inp, t, lid)
        for (j, e, g, u, h, y) in parts:
            p = t * s.k + j
            r = int(np.nonzero(sorted_ids[:ntp] == p)[0][0])
            h_or = bf16_bits_to_f64(h_rows[r])
            # h within one bf16 ulp (the fp32 accumulation can flip a rounding)
            ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(h), 1e-30))[1] - 8)
            if np.any(np.abs(h_or - h) > ulp * 1.0001):
                ok = False
            # y from the oracle's own h, fp64
            W2 = dequant_f64(inp.w2_q[e], inp.w2_s[e])
            y64 = W2 @ h_or
            bound = 1e-5 * (np.abs(W2) @ np.abs(h_or)) + 1e-30
            if np.any(np.abs(y_pairs[p] - y64) > bound):
                ok = False
        # the oracle output is the bf16 rounding of the exact value, up to fp32
        # accumulation error
        worst = max(worst, rounding_ratio(got[t], ref))
    ok = ok and worst <= 1.0
    return ok, f"brute force worst ratio {worst:.3g}"


def pin_topk1_identity(seed=21):
    """k = 1 with weight 1: the layer output is bf16 of that expert's MLP output."""
    inp = small_random_inputs(seed, k=1, emap=False, El=6, Eg=6)
    inp.topk_weights[:] = 1.0
    s = inp.shape
    _, out = oracle.run_workload(inp)
    got = bf16_bits_to_f64(out)
    ok = True
    for t in range(s.T):
        e = int(inp.topk_ids[t, 0])
        W13 = dequant_f64(inp.w13_q[e], inp.w13_s[e])
        W2 = dequant_f64(inp.w2_q[e], inp.w2_s[e])
        x = bf16_bits_to_f64(inp.x[t])
        h = rne_bf16(silu64(W13[:s.I] @ x) * (W13[s.I:] @ x))
        y = W2 @ h
        if rounding_ratio(got[t], y) > 1.0:
            ok = False
    return ok, "top-1 identity"


def pin_token_permutation(seed=31):
    """Permuting tokens permutes output rows bit-exactly."""
    inp = small_random_inputs(seed)
    s = inp.shape
    _, out = oracle.run_workload(inp)
    perm = np.random.default_rng(seed + 1).permutation(s.T)
    inp2 = synth.MoEInputs(s, inp.x[perm], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                           inp.topk_ids[perm], inp.topk_weights[perm], inp.expert_map)
    _, out2 = oracle.run_workload(inp2)
    return bool(np.array_equal(out[perm], out2)), "token permutation changed outputs"


def pin_cross_layout(seed=41):
    """Indexed, grouped-contiguous and grouped-masked layers agree bit-exactly on
    the same draw (per-row outputs and token outputs)."""
    return _cross_layout(small_random_inputs(seed))


def pin_cross_layout_mxfp4(seed=43):
    """The same agreement with MXFP4 weights."""
    inp = small_random_inputs(seed)
    s = inp.shape
    rng = np.random.default_rng(seed + 1)
    inp.w13_s = synth.mx_scales(rng, s.E_local, 2 * s.I, s.H, center=124)
    inp.w2_s = synth.mx_scales(rng, s.E_local, s.H, s.I, center=124)
    with oracle.weight_format("mxfp4"):
        return _cross_layout(inp)


def _cross_layout(inp):
    s = inp.shape
    _, (out, h_rows, y_pairs) = oracle.run_workload(inp, want_h=True, want_y=True)
    a2, m_idx, r2p = synth.grouped_contiguous_layout(inp, align=8)
    rows_c, tok_c = oracle.moe_grouped("contiguous", a2, inp.w13_q, inp.w13_s, inp.w2_q,
                                       inp.w2_s, m_indices=m_idx, row_to_pair=r2p,
                                       topk_weights=inp.topk_weights, T=s.T, k=s.k)
    a3, mm, r2p3 = synth.grouped_masked_layout(inp)
    rows_m, tok_m = oracle.moe_grouped("masked", a3, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                       masked_m=mm, row_to_pair=r2p3,
                                       topk_weights=inp.topk_weights, T=s.T, k=s.k)
    ok = np.array_equal(tok_c, out) and np.array_equal(tok_m, out)
    valid = r2p >= 0
    ok &= np.array_equal(rows_c[valid], f64_to_bf16_bits(rne_bf16(y_pairs[r2p[valid]])))
    v3 = r2p3 >= 0
    ok &= np.array_equal(rows_m[v3], f64_to_bf16_bits(rne_bf16(y_pairs[r2p3[v3]])))
    return bool(ok), "ok" if ok else "layouts disagree"


def check_align(topk_ids, E_global, expert_map, E_local, bm, sorted_ids, expert_ids, ntp):
    """Routing invariants of the aligned layout.  Returns a list of failures."""
    T, k = topk_ids.shape
    P = T * k
    sent = P
    fails = []
    flat = topk_ids.reshape(-1)
    lid = np.full(P, -1)
    for p in range(P):
        g = int(flat[p])
        if 0 <= g < E_global:
            l = g if expert_map is None else int(expert_map[g])
            if 0 <= l < E_local:
                lid[p] = l
    counts = np.bincount(lid[lid >= 0], minlength=E_local)
    want_ntp = int(sum(-(-c // bm) * bm for c in counts))
    if ntp != want_ntp:
        fails.append(f"ntp {ntp} != {want_ntp}")
    cap = sorted_ids.size
    if ntp > cap or ntp % bm:
        fails.append("ntp beyond capacity or not a block multiple")
        return fails
    body = sorted_ids[:ntp]
    real = body[body != sent]
    if not np.array_equal(np.sort(real), np.nonzero(lid >= 0)[0]):
        fails.append("local pairs are not each present exactly once")
    if np.any(sorted_ids[ntp:] != sent):
        fails.append("tail is not the sentinel")
    if np.any((body < 0) | (body > sent)):
        fails.append("out-of-range pair id")
    nb = ntp // bm
    if np.any(expert_ids[nb:] != -1):
        fails.append("expert_ids tail is not -1")
    eb = expert_ids[:nb]
    if nb and (np.any(np.diff(eb) < 0) or eb.min() < 0 or eb.max() >= E_local):
        fails.append("expert_ids not ascending / in range")
    pos = 0
    for e in range(E_local):
        c = counts[e]
        if c == 0:
            if np.any(eb == e):
                fails.append(f"empty expert {e} has a block")
            continue
        seg = -(-c // bm) * bm
        blk = eb[pos // bm:(pos + seg) // bm]
        if blk.size != seg // bm or np.any(blk != e):
            fails.append(f"expert {e} blocks wrong")
        part = sorted_ids[pos:pos + seg]
        want = np.nonzero(lid == e)[0]
        if not np.array_equal(part[:c], want):
            fails.append(f"expert {e} pairs not ascending")
        if np.any(part[c:] != sent):
            fails.append(f"expert {e} padding not sentinel")
        pos += seg
    return fails


def pin_align_invariants(seed=0, n=40):
    rng = np.random.default_rng(seed)
    for it in range(n):
        T = int(rng.integers(0, 40))
        k = int(rng.integers(1, 5))
        Eg = int(rng.integers(k, 20))
        El = int(rng.integers(1, Eg + 1))
        bm = int(rng.choice([1, 2, 4, 8, 16]))
        ids = np.stack([rng.permutation(Eg)[:k] for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        emap = None
        if rng.random() < 0.6:
            emap = np.full(Eg, -1, np.int32)
            emap[rng.permutation(Eg)[:El]] = np.arange(El, dtype=np.int32)
        else:
            El = Eg
        si, ei, ntp = oracle.moe_align(ids, Eg, emap, El, bm)
        f = check_align(ids, Eg, emap, El, bm, si, ei, ntp)
        if f:
            return False, f"draw {it}: {f[:3]}"
        # token permutation: pair sets per expert follow the relabelling
        if T > 1:
            perm = rng.permutation(T)
            si2, ei2, ntp2 = oracle.moe_align(ids[perm], Eg, emap, El, bm)
            if ntp2 != ntp or not np.array_equal(ei2, ei):
                return False, "token permutation changed the block structure"
            body = si[:ntp]
            body2 = si2[:ntp]
            real2 = body2[body2 != T * k]
            # new token i is old token perm[i]
            relabel = perm[real2 // k] * k + real2 % k
            if not np.array_equal(np.sort(relabel), np.sort(body[body != T * k])):
                return False, "token permutation changed the pair set"
    return True, ""


def pin_silu():
    """silu(0) = 0; fp32 silu within 4 fp32 ulps of the fp64 definition over
    a wide range; silu(v) -> v for large v and -> 0 for very negative v."""
    if oracle.silu(0.0) != 0.0:
        return False, "silu(0) != 0"
    vs = np.concatenate([np.linspace(-30, 30, 2001), [-1e-3, 1e-3, 0.5, -0.5, 80.0, -80.0]])
    worst = 0.0
    for v in vs:
        v32 = float(np.float32(v))
        got = oracle.silu(v32)
        want = float(silu64(v32))
        ulp = np.spacing(np.float32(abs(want))) if want != 0 else np.float32(1e-45)
        worst = max(worst, abs(got - want) / float(ulp))
    if abs(oracle.silu(50.0) - 50.0) > 1e-5 or abs(oracle.silu(-50.0)) > 1e-18:
        return False, "silu tails"
    return worst <= 4.0, f"silu worst {worst:.2f} ulp"


def _route_brute(logits, k, renormalize):
    """Router by the definition, written differently from the oracle: the k
    largest logits by a full sort on (-logit, id); the weights from Python
    fp64 exponentials of the shifted logits."""
    import math
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    for t in range(T):
        row = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-row[e], e))[:k]
        m = max(row)
        ex = [math.exp(v - m) for v in row]
        den = sum(ex[e] for e in order) if renormalize else math.fsum(ex)
        ids[t] = order
        w[t] = [ex[e] / den for e in order]
    return ids, w


def pin_route_brute_force(seed=51):
    """Router vs a brute-force sort on small integer-valued logits (many ties),
    with and without renormalisation: ids exactly, weights within 1 fp32 ulp of
    the fp64 value."""
    rng = np.random.default_rng(seed)
    for E, k in [(6, 2), (9, 4), (16, 16), (40, 8), (1, 1)]:
        lg = rng.integers(-3, 4, size=(17, E)).astype(np.float32)
        lg[0, :] = 1.0  # one token with every logit equal
        for renorm in (True, False):
            ids, w = oracle.route_topk(lg, k, renorm)
            bids, bw = _route_brute(lg, k, renorm)
            if not np.array_equal(ids, bids):
                return False, f"ids differ E={E} k={k} renorm={renorm}"
            err = np.abs(w.astype(np.float64) - bw) / np.spacing(np.float32(bw)).astype(np.float64)
            if err.max() > 1.0:
                return False, f"weights off by {err.max():.2f} ulp E={E} k={k} renorm={renorm}"
    return True, "ok"


def pin_route_closed_forms():
    """Closed forms: equal logits give the k lowest ids with weight 1/k
    (renormalised) or 1/E (not); logits ln 2 / 0 give weights 2/3, 1/3 over a
    pair; a constant shift of every logit changes nothing."""
    E, k = 8, 3
    lg = np.zeros((1, E), np.float32)
    ids, w = oracle.route_topk(lg, k, True)
    if list(ids[0]) != [0, 1, 2] or not np.allclose(w, 1.0 / k, rtol=0, atol=1e-7):
        return False, f"equal logits renorm {ids} {w}"
    ids, w = oracle.route_topk(lg, k, False)
    if not np.allclose(w, 1.0 / E, rtol=0, atol=1e-8):
        return False, f"equal logits softmax {w}"
    lg = np.array([[0.0, np.log(2.0), -30.0, -30.0]], np.float32)
    ids, w = oracle.route_topk(lg, 2, True)
    l1 = float(np.float32(np.log(2.0)))
    want = np.array([np.exp(l1) / (np.exp(l1) + 1.0), 1.0 / (np.exp(l1) + 1.0)])
    if list(ids[0]) != [1, 0] or np.abs(w[0] - want).max() > 1e-7:
        return False, f"two-level {ids} {w}"
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((11, 24)).astype(np.float32)
    a = oracle.route_topk(lg, 5, True)
    b = oracle.route_topk(lg + np.float32(16.0), 5, True)
    if not np.array_equal(a[0], b[0]) or np.abs(a[1] - b[1]).max() > 2e-6:
        return False, "shift changed the routing"
    return True, "ok"


def _unpack_codes(w_q):
    """int32 words [..., K/8] -> codes [..., K] (element c = 8w+i in bits 4i..)."""
    u = np.ascontiguousarray(w_q).view(np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    return ((u[..., None] >> shifts) & 0xF).reshape(*u.shape[:-1], u.shape[-1] * 8)


def _pack_positions(kind, E, N, K):
    """Byte position and nibble of every code (e, n, k), and byte position of
    every scale (e, n, g), in the packed buffer, from the format statement
    element by element (the oracle instead walks blocks and copies pieces)."""
    e, n, k = np.meshgrid(np.arange(E), np.arange(N), np.arange(K), indexing="ij")
    if kind == 1:
        up = n >= N // 2
        nn = np.where(up, n - N // 2, n)
        t, r = nn // 64, nn % 64 + np.where(up, 64, 0)
    else:
        t, r = n // 128, n % 128
    KB = (K + 255) // 256  # blocks of a tile (a 128 tail is half a block)
    j, h, c, m = k // 256, (k % 256) // 128, (k % 128) // 32, k % 32
    block = 256 + ((e * (N // 128) + t) * KB + j) * 18432
    byte = block + h * 8192 + r * 64 + (c ^ ((r >> 1) & 3)) * 16 + (m // 8) * 4 + (m % 8) // 2
    high = (m % 2) == 1
    gs = np.arange(K // 32)
    eg, ng, gg = np.meshgrid(np.arange(E), np.arange(N), gs, indexing="ij")
    if kind == 1:
        upg = ng >= N // 2
        nng = np.where(upg, ng - N // 2, ng)
        tg, rg = nng // 64, nng % 64 + np.where(upg, 64, 0)
    else:
        tg, rg = ng // 128, ng % 128
    sblock = 256 + ((eg * (N // 128) + tg) * KB + gg // 8) * 18432
    sbyte = sblock + 16384 + rg * 16 + (gg % 8) * 2
    return byte, high, sbyte


def pin_prepack_positions(seed=61):
    """Every code and scale is where the packed format puts it, for both
    kinds, with random codes and scales: read back through the per-element
    position map, the packed buffer gives the input codes and scales exactly.
    With K % 256 == 128 (the last block half past K) every byte the map does
    not reach, the tail halves included, is zero."""
    rng = np.random.default_rng(seed)
    for kind, (E, N, K) in [(1, (2, 256, 512)), (2, (3, 128, 768)), (1, (1, 384, 256)),
                            (2, (2, 256, 384)), (1, (1, 256, 128))]:
        w_q = rng.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint32).view(np.int32)
        w_s = rng.integers(0, 2**16, size=(E, N, K // 32), dtype=np.uint16)
        out = oracle.prepack(kind, w_q, w_s)
        if out.size != 256 + E * (N // 128) * ((K + 255) // 256) * 18432:
            return False, f"size {out.size}"
        byte, high, sbyte = _pack_positions(kind, E, N, K)
        got = np.where(high, out[byte] >> 4, out[byte] & 0xF)
        if not np.array_equal(got, _unpack_codes(w_q)):
            return False, f"codes misplaced (kind {kind}, {E}x{N}x{K})"
        sg = out[sbyte].astype(np.uint16) | (out[sbyte + 1].astype(np.uint16) << 8)
        if not np.array_equal(sg, w_s):
            return False, f"scales misplaced (kind {kind}, {E}x{N}x{K})"
        covered = np.zeros(out.size, bool)
        covered[:256] = True
        covered[byte.ravel()] = True
        covered[sbyte.ravel()] = True
        covered[sbyte.ravel() + 1] = True
        if out[~covered].any():
            return False, f"bytes outside the map are not zero (kind {kind}, {E}x{N}x{K})"
    return True, "ok"


def pin_prepack_header_and_hand_cases():
    """Header words; the range flag for scales just inside and outside
    [2^-86, 2^35); and three code positions worked out by hand from the
    format (down, E=1, N=128, K=256, every code 0 except one)."""
    w_s = np.full((1, 128, 8), 0x3F80, np.uint16)  # 1.0
    for code_at, want_byte, want_high in [
        # (n=3, k=200): block 0, half 1, row 3, piece (200-128)//32 = 2 stored at
        # 2 ^ ((3 >> 1) & 3) = 3, element 8 of the piece: word 1, low nibble
        # -> 256 + 8192 + 3*64 + 3*16 + 4 = 8692
        ((3, 200), 8692, False),
        # (n=0, k=1): row 0, piece 0 at 0, element 1: byte 256, high nibble
        ((0, 1), 256, True),
        # (n=127, k=127): half 0, row 127, piece 3 stored at 3 ^ 3 = 0, element
        # 31: word 3, byte 3, high nibble -> 256 + 127*64 + 0 + 12 + 3 = 8399
        ((127, 127), 8399, True),
    ]:
        codes = np.zeros((1, 128, 256), np.uint32)
        codes[0, code_at[0], code_at[1]] = 0xB
        w_q = (codes.reshape(1, 128, 32, 8) << (4 * np.arange(8, dtype=np.uint32))).sum(
            axis=-1, dtype=np.uint64).astype(np.uint32).view(np.int32)
        out = oracle.prepack(2, w_q, w_s)
        nz = np.nonzero(out[256:256 + 16384])[0]
        if list(nz + 256) != [want_byte]:
            return False, f"code at {code_at} landed at bytes {list(nz + 256)}"
        v = out[want_byte]
        if (v >> 4 if want_high else v & 0xF) != 0xB:
            return False, f"code at {code_at}: wrong nibble of byte {want_byte}"
    hd = out[:256].view(np.uint32)
    if list(hd[:8]) != [0x4B504843, 1, 2, 1, 128, 256, 18432, 0] or hd[8:].any():
        return False, f"header {list(hd[:8])}"
    # exponent field 41 (2^-86) and 161 (2^34 * 1.x) are in range, 40 and 162 not;
    # +-0 is in range
    for bits, flag in [(41 << 7, 0), (161 << 7 | 0x7F, 0), (0x8000, 0), (40 << 7, 1), (162 << 7, 1),
                       (0x7F80, 1)]:
        s2 = w_s.copy()
        s2[0, 5, 3] = bits
        hd = oracle.prepack(2, w_q, s2)[:256].view(np.uint32)
        if hd[7] != flag:
            return False, f"scale bits {bits:#06x}: flag {hd[7]} != {flag}"
    return True, "ok"


def pin_mxfp4_dequant_exhaustive():
    """MXFP4 dequant: all 16 E2M1 codes x all 256 E8M0 scale bytes against the
    published value table and 2^(s - 127): finite products exact in bf16,
    overflow to +-inf, s = 255 NaN."""
    K = 256 * 32
    codes = np.repeat(np.arange(16, dtype=np.uint32)[:, None], K, axis=1)
    wq = (codes.reshape(16, K // 8, 8) << (4 * np.arange(8, dtype=np.uint32))).sum(
        axis=-1, dtype=np.uint64).astype(np.uint32).view(np.int32)
    ws = np.repeat(np.arange(256, dtype=np.uint8)[None, :], 16, axis=0)
    with oracle.weight_format("mxfp4"):
        got = oracle.dequant(wq, ws, 16, K).astype(np.float64)
    sgn = np.where(np.arange(16) >= 8, -1.0, 1.0)[:, None]
    mag = np.array(E2M1_VALUES)[np.arange(16) & 7][:, None]
    ex = np.repeat(np.arange(256)[None, :], 32, axis=1)
    want = np.ldexp(sgn * mag, ex - 127)
    bf16_max = float(np.ldexp(2.0 - 2.0 ** -7, 127))
    want = np.where(np.abs(want) > bf16_max, np.copysign(np.inf, want), want)
    nan_cols = ex[0] == 255
    if not np.all(np.isnan(got[:, nan_cols])):
        return False, "scale byte 255 is not NaN"
    ok = np.array_equal(got[:, ~nan_cols], want[:, ~nan_cols])
    if not ok:
        bad = np.argwhere(got[:, ~nan_cols] != want[:, ~nan_cols])[0]
        return False, f"code {bad[0]} scale {bad[1] // 32}: {got[:, ~nan_cols][tuple(bad)]} != " \
                      f"{want[:, ~nan_cols][tuple(bad)]}"
    return True, "ok"


def pin_mxfp4_brute_force(seed=31):
    """A small layer with MXFP4 weights against the per-token fp64 brute force
    on the table-based dequant (the same checks as the INT4 brute force)."""
    inp = small_random_inputs(seed)
    s = inp.shape
    rng = np.random.default_rng(seed + 1)
    inp.w13_s = synth.mx_scales(rng, s.E_local, 2 * s.I, s.H, center=124)
    inp.w2_s = synth.mx_scales(rng, s.E_local, s.H, s.I, center=124)
    lid = synth.local_ids(inp)
    with oracle.weight_format("mxfp4"):
        (sorted_ids, _, ntp), (out, h_rows, _) = oracle.run_workload(inp, want_h=True, want_y=True)
    got = bf16_bits_to_f64(out)
    worst = 0.0
    ok = True
    for t in range(s.T):
        ref, parts = brute_force_token(inp, t, lid, deq=dequant_mx_f64)
        for (j, e, g, u, h, y) in parts:
            r = int(np.nonzero(sorted_ids[:ntp] == t * s.k + j)[0][0])
            ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(h), 1e-30))[1] - 8)
            if np.any(np.abs(bf16_bits_to_f64(h_rows[r]) - h) > ulp * 1.0001):
                ok = False
        worst = max(worst, rounding_ratio(got[t], ref))
    ok = ok and worst <= 1.0
    return ok, f"mxfp4 brute force worst ratio {worst:.3g}"


ALL_PINS = {
    "mxfp4_dequant_exhaustive": pin_mxfp4_dequant_exhaustive,
    "mxfp4_brute_force": pin_mxfp4_brute_force,
    "cross_layout_mxfp4": pin_cross_layout_mxfp4,
    "prepack_positions": pin_prepack_positions,
    "prepack_header_and_hand_cases": pin_prepack_header_and_hand_cases,
    "route_brute_force": pin_route_brute_force,
    "route_closed_forms": pin_route_closed_forms,
    "silu": pin_silu,
    "dequant_exhaustive": pin_dequant_exhaustive,
    "dequant_zero_code": pin_dequant_zero_code,
    "one_hot_structure": pin_one_hot_structure,
    "down_one_hot": pin_down_one_hot,
    "closed_form_equal_codes": pin_closed_form_equal_codes,
    "closed_form_gate_up_order": pin_closed_form_gate_up_order,
    "zero_weights": pin_zero_weights,
    "brute_force": pin_brute_force,
    "topk1_identity": pin_topk1_identity,
    "token_permutation": pin_token_permutation,
    "cross_layout": pin_cross_layout,
    "align_invariants": pin_align_invariants,
}
