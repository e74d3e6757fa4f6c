"""Pins for the oracle's packed KV rows (the f2 row: 584-byte packed FP8 and
384-byte NVFP4 rows with a BF16 query).

The pages give only the row sizes (trtllm_batch_decode_sparse_mla_dsv4,
description, SM120/SM121 paragraph: 584 bytes per token; cake_sparse_mla_
sm120_dsv4_nvfp4_decode, Parameters: kv_cache, 384 bytes per token); the byte
layouts are the oracle's reading (module docstring).  These tests tie the
decoders to the element-format definitions (E2M1 from the OCP MX
specification, UE8M0 = 2^(e - 127), E4M3 and BF16 through torch) and check a
hand-built row value by value, and one attention step through it, in closed
form.
"""
import json
import math
import os

import numpy as np
import torch

import oracle
from oracle import oracle as orc

HERE = os.path.dirname(os.path.abspath(__file__))
LOG2E = 1.0 / math.log(2.0)


def bf16_bytes(vals) -> np.ndarray:
    """Little-endian bytes of the BF16 bits of exactly representable values."""
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float32), torch.tensor(np.asarray(vals, dtype=np.float32)))
    return t.view(torch.int16).numpy().view(np.uint16).view(np.uint8)


def e4m3_code(v: float) -> int:
    t = torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn)
    assert float(t.to(torch.float32)) == v
    return int(t.view(torch.uint8)[0])


def test_e2m1_decode_matches_the_specification_for_every_code():
    spec = json.load(open(os.path.join(HERE, "golden", "e2m1_codes.json")))["values"]
    assert len(spec) == 16
    got = orc.E2M1_TABLE
    assert np.array_equal(got, np.array(spec)) and np.array_equal(np.signbit(got), np.signbit(spec))


def test_ue8m0_is_a_power_of_two_exponent():
    e = np.arange(255, dtype=np.uint8)
    got = orc.ue8m0_to_f64(e)
    assert got[127] == 1.0 and got[128] == 2.0 and got[126] == 0.5 and got[0] == 2.0 ** -127
    assert np.array_equal(got, np.array([math.ldexp(1.0, int(k) - 127) for k in e]))


def packed_fp8_row():
    """A 584-byte row and its values: NoPE dim d of block b = d // 64 holds
    E4M3 code for (1 + (d % 8) / 8) with exponent byte 127 + b - 3; the RoPE
    dims hold i / 4 - 8."""
    row = np.zeros(584, np.uint8)
    want = np.zeros(512)
    for d in range(448):
        v = 1.0 + (d % 8) / 8.0
        row[d] = e4m3_code(v)
        want[d] = v * 2.0 ** (d // 64 - 3)
    for b in range(7):
        row[448 + b] = 127 + b - 3
    rope = np.array([i / 4.0 - 8.0 for i in range(64)])
    row[456:584] = bf16_bytes(rope)
    want[448:] = rope
    return row, want


def nvfp4_row():
    """A 384-byte row and its values: NoPE dim d holds E2M1 code d % 16 (low
    nibble first), block b = d // 16 an E4M3 scale 2^(b % 4 - 1), the row
    scale 0.75; the RoPE dims hold -i / 8."""
    spec = json.load(open(os.path.join(HERE, "golden", "e2m1_codes.json")))["values"]
    row = np.zeros(384, np.uint8)
    want = np.zeros(512)
    for d in range(448):
        code = d % 16
        if d % 2 == 0:
            row[d // 2] |= code
        else:
            row[d // 2] |= code << 4
        want[d] = spec[code] * 2.0 ** (d // 16 % 4 - 1) * 0.75
    for b in range(28):
        row[224 + b] = e4m3_code(2.0 ** (b % 4 - 1))
    rope = np.array([-i / 8.0 for i in range(64)])
    row[252:380] = bf16_bytes(rope)
    row[380:384] = np.frombuffer(np.float32(0.75).tobytes(), np.uint8)
    want[448:] = rope
    return row, want


def test_packed_fp8_row_closed_form():
    row, want = packed_fp8_row()
    got = orc.decode_packed_fp8_rows(row[None])[0]
    assert np.array_equal(got, want)
    assert oracle.PACKED_ROW_BYTES["packed_fp8"] == 584 == 448 + 7 + 1 + 2 * 64


def test_nvfp4_row_closed_form():
    row, want = nvfp4_row()
    got = orc.decode_nvfp4_rows(row[None])[0]
    assert np.array_equal(np.abs(got), np.abs(want)) and np.array_equal(got, want)
    assert oracle.PACKED_ROW_BYTES["nvfp4"] == 384 == 448 // 2 + 448 // 16 + 2 * 64 + 4


def single_slot(dtype, row, want):
    """One token, one valid compressed slot holding ``row``: O = bmm2 * row,
    LSE2 = bmm1 * <q, row> * log2(e) (a BF16 query)."""
    H = 3
    rng = np.random.default_rng(7)
    q = torch.tensor(rng.standard_normal((1, H, 512)).astype(np.float32)).to(torch.bfloat16)
    qd = q.to(torch.float64).numpy()[0]
    qbits = q.view(torch.int16).numpy().view(np.uint16)
    nbytes = row.shape[0]
    swa = np.zeros((2, nbytes), np.uint8)
    comp = np.zeros((4, nbytes), np.uint8)
    comp[2] = row
    idx = np.full((1, 130), -1, np.int32)
    idx[0, 129] = 2
    bmm1, bmm2 = 0.04, 1.25
    o, lse = orc.sparse_mla_decode(dtype=dtype, batch=1, q=qbits, swa_kv=swa, comp_kv=comp, indices=idx,
                                   seq_lens=np.array([1000], np.int32), bmm1_scale=bmm1, bmm2_scale=bmm2)
    np.testing.assert_allclose(o[0], bmm2 * np.tile(want, (H, 1)), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse[0], bmm1 * (qd @ want) * LOG2E, rtol=1e-12, atol=1e-12)


def test_single_slot_through_a_packed_fp8_row():
    single_slot("packed_fp8", *packed_fp8_row())


def test_single_slot_through_an_nvfp4_row():
    single_slot("nvfp4", *nvfp4_row())
