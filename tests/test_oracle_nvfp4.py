"""Pins of the oracle's two-level NVFP4 quantizer (1x16 E2M1 blocks, an E4M3
block scale, an FP32 scale per token / group / tensor) against hand-worked
rows, exact round trips, format bounds and the batch-composition invariance
that motivates per-token scaling."""
import numpy as np
import torch

import oracle
from moe_mx8_quantize_gb300 import inputs


def bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(vals, dtype=torch.float32)), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def test_worked_row():
    """A 32-element token with amax 384 = 2688/7, so S_enc = 2688/384 = 7
    exactly and S_dec = RN(384/2688) = RN(1/7) (bits 0x3E124925).

    Block 0 (amax 384): 384/6 = 64, *7 = 448 -> block scale 448 (0x7E);
      r = 7/448 = 1/64 exactly, so x*r is exact:
        384->6 (7)  -192->-3 (0xD)  96->1.5 (3)  16->0.25 tie->0 (0)
        48->0.75 tie->1 (2)  80->1.25 tie->1 (2)  112->1.75 tie->2 (4)
        160->2.5 tie->2 (4)  224->3.5 tie->4 (6)  320->5 tie->4 (6)
        -16->-0.25 tie->-0 (8)  0->0 (0)  -0->-0 (8)  1->1/64->0 (0)
        200->3.125->3 (5)  32->0.5 (1)
    Block 1 (amax 12): 12/6 = 2, *7 = 14 -> block scale 14 (0x56); r = 7/14 = 0.5:
        12->6 (7)  -12->-6 (0xF)  5->2.5 tie->2 (4)  7->3.5 tie->4 (6)
        3->1.5 (3)  0.5->0.25 tie->0 (0)  1.5->0.75 tie->1 (2)
        2.5->1.25 tie->1 (2)  3.5->1.75 tie->2 (4)  10->5 tie->4 (6)
        9->4.5->4 (6)  11->5.5->6 (7)  -1->-0.5 (9)  2->1 (2)  4->2 (4)  8->4 (6)
    Element 2j is the low nibble of byte j."""
    b0 = [384, -192, 96, 16, 48, 80, 112, 160, 224, 320, -16, 0, -0.0, 1, 200, 32]
    b1 = [12, -12, 5, 7, 3, 0.5, 1.5, 2.5, 3.5, 10, 9, 11, -1, 2, 4, 8]
    x = bf16_bits([float(v) for v in b0 + b1]).reshape(1, 32)
    x[0, 12] = 0x8000  # make sure the -0.0 entry is the negative zero pattern
    q, s, s32 = oracle.nvfp4_quantize(x)
    assert s.tolist() == [[0x7E, 0x56]]
    assert s32.view(np.uint32).tolist() == [0x3E124925]
    assert q[0].tolist() == [0xD7, 0x03, 0x22, 0x44, 0x66, 0x08, 0x08, 0x15,
                             0xF7, 0x64, 0x03, 0x22, 0x64, 0x76, 0x29, 0x64]


def test_zero_row_and_tiny_row_are_finite():
    x = np.zeros((2, 32), np.uint16)
    x[1, 3] = 0x0001          # a single bf16 subnormal: S_enc clamps to FLT_MAX
    x[1, 7] = 0x8001
    q, s, s32 = oracle.nvfp4_quantize(x)
    assert (q[0] == 0).all() and (s[0] == 0).all() and s32[0] == 0.0
    assert np.isfinite(s32).all()
    d = oracle.dequant_nvfp4(q, s, s32)
    assert np.isfinite(d).all()
    assert (s != 0x7F).all() and (s != 0xFF).all()


def _exact_rows(rng, R, C, j_range=(-20, 20)):
    """Rows whose amax is 2688*2^j (S_enc = 2^-j, S_dec = 2^j exactly) built from
    blocks e2m1 * sb * 2^j where sb is an E4M3 value and each block holds
    6*sb*2^j, and the row holds 6*448*2^j once."""
    grid = np.array([oracle.e2m1_decode(c) for c in range(16)])
    e4 = np.array([oracle.e4m3_decode(c) for c in range(1, 127)])
    nb = C // 16
    j = rng.integers(*j_range, size=(R, 1))
    sb = e4[rng.integers(0, e4.size, size=(R, nb))]
    sb[:, 0] = 448.0
    codes = rng.integers(0, 16, size=(R, C))
    codes[:, ::16] = 7
    vals = grid[codes] * np.repeat(sb, 16, axis=1) * np.exp2(j)
    return vals.astype(np.float32)


def test_round_trip_of_representable_rows():
    rng = np.random.default_rng(7)
    xf = _exact_rows(rng, 64, 256)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    if not torch.equal(x.float(), torch.from_numpy(xf)):
        keep = (x.float() == torch.from_numpy(xf)).all(1)
        xf, x = xf[keep.numpy()], x[keep]
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s, s32 = oracle.nvfp4_quantize(xb)
    d = oracle.dequant_nvfp4(q, s, s32)
    assert np.array_equal(d, xf)


def test_block_codes_bounded_and_error_bound():
    x = inputs.bits(inputs.pr1()["X"])
    q, s, s32 = oracle.nvfp4_quantize(x)
    assert ((s & 0x80) == 0).all() and (s != 0x7F).all()
    sbv = np.array([oracle.e4m3_decode(int(c)) for c in range(256)])[s]
    assert (sbv <= 448).all()
    d = oracle.dequant_nvfp4(q, s, s32).astype(np.float64)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    # each element is within one E2M1 grid step (<= 2) of its scaled value:
    # |x^ - x| <= 1.0 * sb * S_dec, with slack for the FP32 scale chain
    bound = np.repeat(sbv, 16, axis=1) * s32[:, None].astype(np.float64)
    assert (np.abs(d - xf) <= bound * (1 + 1e-5) + 1e-30).all()
    # the amax of each token lands on +-6 * sb * S_dec with sb close to 448
    amax_col = np.abs(xf).argmax(1)
    codes = np.where(amax_col % 2 == 0, q[np.arange(len(q)), amax_col // 2] & 15,
                     q[np.arange(len(q)), amax_col // 2] >> 4)
    assert ((codes & 7) == 7).all()


def test_per_token_invariance_to_batch_composition():
    """A token's bytes and FP32 scale do not depend on which other tokens are
    in the batch, their order or their number (per-token scaling: Miles page,
    "Un Cuantizador Compartido Es el Mecanismo Real")."""
    x = inputs.bits(inputs.qwen_moe(with_weights=False, tokens=96, hidden=256)["X"])
    q, s, s32 = oracle.nvfp4_quantize(x)
    perm = np.random.default_rng(0).permutation(96)[:40]
    q2, s2, s322 = oracle.nvfp4_quantize(x[perm])
    assert np.array_equal(q2, q[perm]) and np.array_equal(s2, s[perm])
    assert np.array_equal(s322, s32[perm])
    # a token quantized alone
    qa, sa, s32a = oracle.nvfp4_quantize(x[17:18])
    assert np.array_equal(qa[0], q[17]) and s32a[0] == s32[17]
    # a per-tensor scale is batch-variant: adding a large token changes others
    xt = x.copy()
    xt[0] = 0x4780  # 65536.0 everywhere in token 0
    qt, st, s32t = oracle.nvfp4_quantize(xt, scope=oracle.SCOPE_TENSOR)
    qt2, st2, _ = oracle.nvfp4_quantize(x, scope=oracle.SCOPE_TENSOR)
    assert not np.array_equal(qt[1:], qt2[1:])


def test_scope_special_cases():
    x = inputs.bits(inputs.pr1()["W"])[:64]
    q_tok, s_tok, s32_tok = oracle.nvfp4_quantize(x)
    # groups of one row reproduce per-token scaling
    offs = np.arange(65)
    q_g, s_g, s32_g = oracle.nvfp4_quantize(x, oracle.SCOPE_GROUP, offs)
    assert np.array_equal(q_g, q_tok) and np.array_equal(s_g, s_tok) and np.array_equal(s32_g, s32_tok)
    # one group reproduces per-tensor scaling
    q_t, s_t, s32_t = oracle.nvfp4_quantize(x, oracle.SCOPE_TENSOR)
    q_1, s_1, s32_1 = oracle.nvfp4_quantize(x, oracle.SCOPE_GROUP, [0, 64])
    assert np.array_equal(q_t, q_1) and np.array_equal(s_t, s_1) and np.array_equal(s32_t, s32_1)
    # empty groups are allowed and give a zero decode scale
    q_e, s_e, s32_e = oracle.nvfp4_quantize(x, oracle.SCOPE_GROUP, [0, 0, 30, 30, 64])
    assert s32_e[0] == 0.0 and s32_e[2] == 0.0
    qa, sa, _ = oracle.nvfp4_quantize(x[:30], oracle.SCOPE_TENSOR)
    assert np.array_equal(q_e[:30], qa) and np.array_equal(s_e[:30], sa)


def test_fp32_scale_is_the_token_amax_over_2688():
    x = inputs.bits(inputs.pr1()["X"])
    _, _, s32 = oracle.nvfp4_quantize(x)
    amax = np.abs(oracle.bf16_to_f32(x)).max(1)
    # S_dec = RN_f32(amax / 2688): compare with the correctly rounded quotient
    exact = amax.astype(np.float64) / 2688.0
    assert np.array_equal(s32, exact.astype(np.float32))


def test_quantize_before_dispatch_is_bit_identical():
    """Per-token scaling makes the codes of a token independent of the batch:
    quantizing the MoE-dispatched rows (each token repeated top-k times,
    grouped by expert) gives the gathered rows of the token-major
    quantization, byte for byte -- the reason the fused MoE GEMM may gather
    tokens quantized once before dispatch."""
    from moe_mx8_quantize_gb300 import inputs
    d = inputs.moe(4, "cpu", 96, 256, 6, 128, 3, with_weights=False)
    tor = inputs.dispatch(d["topk_ids"], 6).token_of_row.numpy()
    Xb = inputs.bits(d["X"])
    q, s, t = oracle.nvfp4_quantize(Xb)
    q2, s2, t2 = oracle.nvfp4_quantize(Xb[tor])
    assert len(tor) == 96 * 3
    assert np.array_equal(q2, q[tor]) and np.array_equal(s2, s[tor])
    assert np.array_equal(t2.view(np.uint32), t[tor].view(np.uint32))
