"""Write oracle_hashes.json: SHA-256 of the oracle's outputs on small seeded cases.

Calls only the CPU oracle and the seeded input generators.  The stored hashes
pin the oracle against accidental drift (the A/B output-hash comparison of the
prhub.com.cn digest of SGLang PR #34085, section 讨论亮点, applied to the
oracle itself).  Re-run only for a change to the oracle's arithmetic that a
passage of the pages, or a reading of one, justifies.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def cases():
    d = synth.tiny_ln_modulate()
    x = u16(d["x"]).reshape(-1, 512)
    yield "tiny.ln_modulate", oracle.ln_modulate(x, u16(d["scale"]), u16(d["shift"]), 1e-6)
    yield "tiny.rmsnorm_scale", oracle.rmsnorm_scale(x, u16(d["weight"]), u16(d["scale"]), 1e-6)
    s = synth.sweep_case(1024, 77)
    xs = u16(s["x"].contiguous())
    yield "sweep1024x77.rmsnorm_tanh_residual", oracle.rmsnorm_tanh_residual(
        xs, u16(s["gate_tok"].contiguous()), u16(s["residual"].contiguous()), u16(s["weight"]), 1e-6)
    yield "sweep1024x77.residual_gate_add", oracle.residual_gate_add(
        xs, u16(s["gate"].contiguous()), u16(s["y"].contiguous()))
    q = synth.qkv_epilogue_case(batch=2, s_txt=8, grid_h=4, grid_w=6, heads=4)
    yield "qkv_small.joint", oracle.qkv_epilogue(
        u16(q["txt"]), u16(q["img"]), q["batch"], q["heads"], q["head_dim"],
        u16(q["wq_txt"]), u16(q["wk_txt"]), u16(q["wq_img"]), u16(q["wk_img"]),
        q["cos_txt"].numpy(), q["sin_txt"].numpy(), q["cos_img"].numpy(), q["sin_img"].numpy(), 1e-6)
    yield "tanh_bf16.table", oracle.tanh_table()


def compute():
    return {k: hashlib.sha256(np.ascontiguousarray(v).tobytes()).hexdigest() for k, v in cases()}


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_hashes.json"), "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
        f.write("\n")
