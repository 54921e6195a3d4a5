"""MXFP4 weights on the GPU (chord_mxfp4_prepack + CHORD_FLAG_MXFP4).

The MXFP4 variant of the layer (vLLM Kimi K3 production support page, "MXFP4
MoE"; OCP Microscaling FP4): E2M1 codes with one E8M0 scale byte per 32 input
channels, w = bf16(e2m1(q) * 2^(e - 127)), the rest of the layer as for INT4.

  * The pack is a byte rearrangement plus the widening of each scale byte to
    the bf16 value 2^(e - 127): the GPU's pack must equal the oracle's pack of
    the same codes with those bf16 scales (widened here from the definition,
    independently of the library) byte for byte, header format word included.
  * Every code x every scale byte: a one-hot intermediate h (gate weight 4 and
    up weight 0.5 on one input channel of value 4 give h = bf16(silu(16) * 2)
    = 32 exactly on one channel, 0 elsewhere) makes each grouped row output
    bf16(32 * W2[:, i0]), so whole columns of the down weight are read back.
    Row n of W2 takes scale byte n (0..255) and code n % 16 in that column:
    both the one-multiply dequant (bytes <= 128) and the split multiply
    (bytes > 128) run, and the outputs must equal the oracle's bit for bit
    (NaN where it is NaN) and 32 * e2m1 * 2^(e - 127) from the E2M1 table.
  * Whole layers (indexed, masked, contiguous) against the oracle with the
    same split check and fp64 anchor as the INT4 layer."""

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_util import dev_tensor
from test_gpu_layer import (DEV, chord, masked_layer_check, run_indexed_full,  # noqa: F401
                            small, verify_indexed)
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def widen_e8m0(s8: np.ndarray) -> np.ndarray:
    """bf16 bits of 2^(e - 127) for E8M0 bytes e (NaN 0x7FC0 for 255), from the
    definition: rne_bf16 of the power of two, which is exact."""
    e = s8.astype(np.int64)
    v = np.ldexp(1.0, np.where(e == 255, 0, e) - 127)
    bits = pins.f64_to_bf16_bits(pins.rne_bf16(v)).astype(np.uint16)
    return np.where(e == 255, np.uint16(0x7FC0), bits).astype(np.uint16)


def mx_weights(inp):
    """Device tensors of an MXFP4 draw: codes int32 and scale bytes uint8."""
    return (dev_tensor(inp.w13_q, DEV), dev_tensor(inp.w13_s, DEV), dev_tensor(inp.w2_q, DEV),
            dev_tensor(inp.w2_s, DEV))


def mx_small(T, k, Eg, El, H, I, seed, emap=True, center=121):
    inp = small(T, k, Eg, El, H, I, seed, emap=emap)
    rng = np.random.default_rng(seed + 7)
    inp.w13_s = synth.mx_scales(rng, El, 2 * I, H, center=center)
    inp.w2_s = synth.mx_scales(rng, El, H, I, center=center)
    return inp


@pytest.mark.parametrize("kind,E,N,K", [(1, 2, 256, 512), (2, 3, 256, 256), (2, 1, 384, 2048),
                                        (2, 3, 256, 384)])
def test_mxfp4_pack_matches_oracle(chord, kind, E, N, K):
    rng = np.random.default_rng(E * 100 + N + K + kind)
    w_q = rng.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint32).view(np.int32)
    s8 = rng.integers(0, 256, size=(E, N, K // 32)).astype(np.uint8)
    s8.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)  # every byte at least once
    got = chord.prepack(dev_tensor(w_q, DEV), dev_tensor(s8, DEV), kind).cpu().numpy()
    ref = oracle.prepack(kind, w_q, widen_e8m0(s8))
    hdr = ref[:256].view(np.uint32).copy()
    hdr[7] = 0  # an MXFP4 pack records no INT4 scale-range flag
    hdr[8] = 1  # weight format: MXFP4
    ref[:256] = hdr.view(np.uint8)
    assert got.size == ref.size == chord.prepack_size(kind, E, N, K)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


def test_mxfp4_every_code_and_scale_byte(chord):
    E, H, I = 1, 256, 256
    c0, i0 = 37, 70  # input channel, intermediate channel (group i0 // 32 = 2)
    c13 = np.zeros((E, 2 * I, H), np.int64)  # code 0: +0.0
    c13[0, i0, c0] = 6        # e2m1 0b0110 = 4.0: gate = 4 * x
    c13[0, I + i0, c0] = 1    # e2m1 0b0001 = 0.5: up = 0.5 * x
    s13 = np.full((E, 2 * I, H // 32), 127, np.uint8)  # 2^0
    rng = np.random.default_rng(3)
    c2 = rng.integers(0, 16, size=(E, H, I))
    # the rest of column i0's scale group is +0 (so no overflowing weight there
    # meets h = 0 and makes a NaN); the other groups (scale 1) are random
    g0 = i0 // 32 * 32
    c2[0, :, g0:g0 + 32] = 0
    c2[0, :, i0] = np.arange(H) % 16
    s2 = np.full((E, H, I // 32), 127, np.uint8)
    s2[0, :, i0 // 32] = np.arange(H, dtype=np.uint8)  # row n: scale byte n
    w13_q, w2_q = synth.pack_codes(c13), synth.pack_codes(c2)
    M = 16
    a = np.zeros((M, H), np.uint16)
    a[0, c0] = 0x4080  # 4.0
    m_idx = np.full(M, -1, np.int32)
    m_idx[0] = 0
    pw = chord.prepack_weights(dev_tensor(w13_q, DEV), dev_tensor(s13, DEV),
                               dev_tensor(w2_q, DEV), dev_tensor(s2, DEV))
    h = torch.empty((M, I), dtype=torch.bfloat16, device=DEV)
    rows = chord.w4a16_moe_grouped("contiguous", dev_tensor(a, DEV, True), pw, None, None, None,
                                   m_indices=dev_tensor(m_idx, DEV), flags=1, h_out=h)
    torch.cuda.synchronize()
    h0 = pins.bf16_bits_to_f64(h[0].view(torch.int16).cpu().numpy().view(np.uint16))
    want_h = np.zeros(I)
    want_h[i0] = 32.0
    assert np.array_equal(h0, want_h), "the intermediate is not the one-hot 32"
    got = rows[0].view(torch.int16).cpu().numpy().view(np.uint16)
    with oracle.weight_format("mxfp4"):
        ref_rows = oracle.moe_grouped("contiguous", a, w13_q, s13, w2_q, s2, m_indices=m_idx)
    ref = ref_rows[0]
    g, r = pins.bf16_bits_to_f64(got), pins.bf16_bits_to_f64(ref)
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan), "NaN pattern differs from the oracle"
    assert np.array_equal(got[~nan], ref[~nan]), "column values differ from the oracle"
    # and from the E2M1 table: 32 * e2m1(n % 16) * 2^(n - 127), bf16-rounded
    n = np.arange(H)
    code = n % 16
    val = np.where(code >= 8, -1.0, 1.0) * np.array(pins.E2M1_VALUES)[code & 7]
    want = pins.rne_bf16(np.ldexp(32.0 * val, n - 127))
    fin = n < 255
    assert np.array_equal(g[fin], want[fin]), "column values differ from the E2M1 table"
    assert np.all(np.isnan(g[255])), "scale byte 255 must give NaN"


def _mx_verify(chord, inp, tokens=None, label=""):
    w = mx_weights(inp)
    pw = chord.prepack_weights(*w)
    with oracle.weight_format("mxfp4"):
        run = run_indexed_full(chord, inp, weights=(pw, None, None, None))
        return verify_indexed(inp, run, tokens, label=label)


@pytest.mark.parametrize("name,args", [
    ("decode-map", (40, 3, 10, 6, 512, 256, 81)),
    ("prefill-tile", (700, 2, 3, 3, 256, 256, 82)),
    ("split-k", (3, 8, 16, 16, 2048, 256, 83)),
    ("decode64", (64, 4, 8, 8, 512, 512, 84)),
    # K = I = 256 is one stage: the 64-token token-stationary down tile
    ("one-stage-down64", (64, 4, 8, 8, 512, 256, 88)),
    # about 60 rows per expert: the 128-token tile
    ("decode128", (120, 4, 8, 8, 512, 512, 89)),
])
def test_mxfp4_indexed_small(chord, name, args):
    T, k, Eg, El, H, I, seed = args
    _mx_verify(chord, mx_small(T, k, Eg, El, H, I, seed, emap=El < Eg), label=f"mxfp4 {name}")


def test_mxfp4_large_scale_bytes_in_the_gate_up_gemm(chord):
    """Scale bytes above 128 in the gate/up weights take the split multiply
    there too (weights above 2 times their code)."""
    inp = mx_small(48, 4, 8, 8, 512, 256, 85, emap=False, center=110)
    inp.w13_s[::3, ::5, 1] = 133
    inp.w2_s[1::2, ::7, 0] = 131
    _mx_verify(chord, inp, label="mxfp4 large scale bytes")


def test_mxfp4_masked_and_indexed_agree(chord):
    inp = mx_small(80, 3, 10, 6, 512, 256, 86)
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    pw = chord.prepack_weights(*mx_weights(inp))
    with oracle.weight_format("mxfp4"):
        toks = masked_layer_check(chord, inp, a3, mm, r2p, (pw, None, None, None), "mxfp4 masked")
        ind = run_indexed_full(chord, inp, weights=(pw, None, None, None))
        verify_indexed(inp, ind, label="mxfp4 indexed (same draw)")


def test_mxfp4_ep8_decode(chord):
    """The EP8 decode workload's shapes with MXFP4 weights, sampled tokens."""
    s = synth.workload("ep8-decode")
    inp = synth.make_inputs(s, weight_format="mxfp4")
    tokens = np.random.default_rng(8).choice(s.T, 48, replace=False)
    _mx_verify(chord, inp, tokens, label="mxfp4 EP8 decode T=512 (48 sampled tokens)")


def test_mxfp4_tp8_t128(chord):
    """The TP8 shapes (384 experts, H = 7168, I = 256) with MXFP4 weights at
    T = 128: the one-stage down GEMM runs token-stationary units of several
    weight tiles each; sampled tokens."""
    s = synth.workload("tp8", T=128)
    inp = synth.make_inputs(s, weight_format="mxfp4")
    tokens = np.random.default_rng(9).choice(s.T, 32, replace=False)
    _mx_verify(chord, inp, tokens, label="mxfp4 TP8 T=128 (32 sampled tokens)")


def test_mxfp4_packs_are_not_int4_packs(chord):
    """An MXFP4 pack passed as INT4 (and the reverse) is refused by the header
    check: nothing is computed and CHORD_ERR_PACKED is reported."""
    inp = mx_small(16, 2, 4, 4, 256, 256, 87, emap=False)
    s = inp.shape
    pw = chord.prepack_weights(*mx_weights(inp))
    pw.fmt = "int4"  # lie about the format
    x = dev_tensor(inp.x, DEV, True)
    ids = dev_tensor(inp.topk_ids, DEV)
    si, ei, ntp = chord.moe_align(ids, s.E_global, s.E_local, 16)
    with pytest.raises(chord.ChordError) as ex:
        chord.w4a16_moe_indexed(x, pw, None, None, None, dev_tensor(inp.topk_weights, DEV), si,
                                ei, ntp, 16, s.E_global, flags=1)
    assert ex.value.status == -11
