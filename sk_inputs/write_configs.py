"""Writes sk_inputs/configs.json: the sequence lengths, query lengths and shapes of
the eight benchmark workloads as the seeded generator produces them, so the
workloads can be read without running anything and a test can check that the
generator still reproduces them.

    python sk_inputs/write_configs.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import sk_inputs as si  # noqa: E402


def describe(index: int) -> dict:
    w = si.config(index)
    return {"index": index, "name": w.name, "seed": w.seed, "bs": int(w.bs),
            "seq_lens": [int(x) for x in w.seq_lens], "q_lens": [int(x) for x in w.q_lens],
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "page": w.page, "kv_dtype": "fp8_e4m3" if w.kv_dtype == si.KV_FP8 else "bf16",
            "k_scale": w.k_scale, "v_scale": w.v_scale, "causal": w.causal, "num_sms_plan": w.num_sms,
            "seg_max": w.seg_max, "kv_bytes": int(w.kv_bytes)}


def main():
    out = {"workloads": [describe(i) for i in range(1, 9)]}
    with open(os.path.join(HERE, "configs.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
