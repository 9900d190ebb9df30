"""Loader for the hand-worked fixtures under tests/golden/ (plain text)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CASES = ["sym_fp16_m2_k16_n8", "asym_fp16_m2_k16_n8", "round_bf16_m1_k16_n8",
         "round_fp16_m1_k16_n8", "lib_sym_fp16_m2_k32_n8"]


def _num(tok):
    return int(tok, 16) if tok.lower().startswith(("0x", "-0x")) else float(tok)


def load(name):
    raw = {}
    with open(os.path.join(GOLDEN, name + ".txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "dtype":
                continue
            raw[key] = [_num(v) for v in vals]
    M, K, N, G = (int(raw[k][0]) for k in ("M", "K", "N", "G"))
    case = dict(name=name, M=M, K=K, N=N, G=G, sym=bool(raw["sym"][0]))
    with open(os.path.join(GOLDEN, name + ".txt")) as f:
        for line in f:
            if line.startswith("dtype"):
                case["dtype"] = 0 if line.split()[1] == "fp16" else 1
    if "q_row" in raw:
        q = np.tile(np.array(raw["q_row"], dtype=np.uint8), (N, 1))
    else:
        q = np.repeat(np.array(raw["q_per_row"], dtype=np.uint8)[:, None], K, axis=1)
    case["q"] = q
    if "qweight_words" in raw:
        case["qweight_words"] = np.array([w & 0xFFFFFFFF for w in raw["qweight_words"]],
                                         dtype=np.uint64)
    if "scales_bits" in raw:
        case["scales_bits"] = np.array(raw["scales_bits"], dtype=np.uint16)[:, None]
    else:
        case["scales_vals"] = np.array(raw["scales"], dtype=np.float64)[:, None]
    if not case["sym"]:
        case["z"] = np.array(raw["zeros"], dtype=np.uint8)[:, None]
        case["qzeros_words"] = np.array(raw["qzeros_words"], dtype=np.uint64)
    case["x_vals"] = np.array([raw[f"x{m}"] for m in range(M)], dtype=np.float64)
    case["y"] = np.array([raw[f"y{m}"] for m in range(M)], dtype=np.float64)
    if "w_bits" in raw:
        case["w_bits"] = np.array(raw["w_bits"], dtype=np.uint16)
    if "y0_exact_weights" in raw:
        case["y_exact"] = np.array([raw["y0_exact_weights"]], dtype=np.float64)
    return case


def to_bits(vals, dtype):
    """Encode exactly-representable values as 16-bit patterns (numpy/torch casts)."""
    vals = np.asarray(vals, dtype=np.float64)
    if dtype == 0:
        return vals.astype(np.float16).view(np.uint16)
    import torch
    t = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)
