"""Fixed values the pages print (tests/golden/, each file cites its page and
section) checked against the oracle, the header, the binding and the input
generator: the model dimensions, and the block structs' sizes and field
offsets (values placed at the printed offsets must be the ones the oracle's
dequantisation reads)."""
import os
import re

import numpy as np

import oracle
import synth
import bit_quantized_moe_bias_b300 as B
from helpers import E, F, H, K

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
HEADER = os.path.join(os.path.dirname(GOLDEN), "..", "include", "ds4g.h")


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _layouts():
    out = {}
    for r in _rows("quant_block_layouts.txt"):
        if r[0].startswith("block_"):
            out[r[0]] = (int(r[1]), {k: (int(o), int(n)) for k, o, n in (f.split(":") for f in r[2:])})
    return out


def test_model_constants():
    c = {k: int(v) for k, v in _rows("ds4_model_constants.txt")}
    assert (H, F, E, K) == (c["N_EMBD"], c["N_FF_EXP"], c["N_EXPERT"], c["N_EXPERT_USED"])
    assert (B.N_EMBD, B.N_FF_EXP, B.N_EXPERT, B.N_EXPERT_USED) == (H, F, E, K)
    text = open(HEADER, encoding="utf-8").read()
    defs = dict(re.findall(r"#define (DS4G_N_[A-Z_]+)\s+(\d+)", text))
    assert int(defs["DS4G_N_EMBD"]) == c["N_EMBD"] and int(defs["DS4G_N_FF_EXP"]) == c["N_FF_EXP"]
    assert int(defs["DS4G_N_EXPERT"]) == c["N_EXPERT"] and int(defs["DS4G_N_EXPERT_USED"]) == c["N_EXPERT_USED"]
    assert c["N_EXPERT_SHARED"] == 1 and c["N_LAYER"] == 43


def test_block_sizes_and_bpw():
    lay = _layouts()
    q2, iq2 = lay["block_q2_K"], lay["block_iq2_xxs"]
    for (total, fields) in (q2, iq2):
        assert sum(n for _, n in fields.values()) == total          # no padding
    assert synth.BLOCK_BYTES[synth.Q2_K] == q2[0] == B.ds4g_block_bytes(synth.Q2_K)
    assert synth.BLOCK_BYTES[synth.IQ2_XXS] == iq2[0] == B.ds4g_block_bytes(synth.IQ2_XXS)
    bpw = {r[1]: float(r[2]) for r in _rows("quant_block_layouts.txt") if r[0] == "bpw"}
    assert abs(iq2[0] * 8 / 256 - bpw["block_iq2_xxs"]) < 0.005
    # the generator writes its fp16 scales exactly where the structs put d / dmin
    assert synth.FP16_FIELDS[synth.Q2_K] == (q2[1]["d"][0], q2[1]["dmin"][0])
    assert synth.FP16_FIELDS[synth.IQ2_XXS] == (iq2[1]["d"][0],)


def _put_f16(block, off, value):
    block[off:off + 2] = np.frombuffer(np.float16(value).tobytes(), np.uint8)


def test_oracle_reads_q2k_fields_at_printed_offsets():
    total, f = _layouts()["block_q2_K"]
    blk = np.zeros(total, np.uint8)
    so, sn = f["scales"]
    qo, qn = f["qs"]
    blk[so:so + sn] = 0x21                       # every sub-block: scale 1, min 2
    blk[qo:qo + qn] = 0xFF                       # every quant 3
    _put_f16(blk, f["d"][0], 2.0)
    _put_f16(blk, f["dmin"][0], 0.25)
    w = oracle.dequantize(synth.Q2_K, blk.reshape(1, -1), 1, 256)
    assert np.all(w == 2.0 * 1 * 3 - 0.25 * 2)   # d * scale * q - dmin * min, each read where printed
    _put_f16(blk, f["dmin"][0], 0.0)
    assert np.all(oracle.dequantize(synth.Q2_K, blk.reshape(1, -1), 1, 256) == 6.0)


def test_oracle_reads_iq2_scale_at_printed_offset():
    total, f = _layouts()["block_iq2_xxs"]
    grid = synth.iq2_grid(0)
    blk = np.zeros(total, np.uint8)
    _put_f16(blk, f["d"][0], 1.0)
    w1 = oracle.dequantize(synth.IQ2_XXS, blk.reshape(1, -1), 1, 256, grid)
    _put_f16(blk, f["d"][0], 2.0)
    w2 = oracle.dequantize(synth.IQ2_XXS, blk.reshape(1, -1), 1, 256, grid)
    assert np.any(w1 != 0) and np.array_equal(w2, 2.0 * w1)     # d scales every weight
    # grid index bytes live in qs (all 0 here: grid row 0 for every group)
    assert np.array_equal(w1[0, :8], 0.125 * grid[0].astype(np.float32))
