"""Writes tests/golden/pair_counts.json using only the oracle (oracle.counts).

The per-(b, h) attended-pair totals and key-index sums of the seven workloads.
Neighbour sets: "pi-Attention: Periodic Sparse Transformers for Efficient
Long-Context Modeling" section 2.1 (causal band [i-k, i]) and 2.2 (skip keys
i - m*pi, m = 1..S, kept when m*pi > k and i - m*pi >= 0); ECP page section 2
(keys of half-segments s-1 and s, causal); bidirectional pi-Attention, the general form of
2.1-2.2 (band [i-k, i+k] and skip keys i -/+ m*pi inside [0, N)).

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

WORKLOADS = {
    "C1": dict(N=256, k_local=16, period=32, S=1, mode=0),
    "C2": dict(N=4096, k_local=128, period=256, S=1, mode=0),
    "C3": dict(N=8192, k_local=512, period=0, S=0, mode=1),
    "C4": dict(N=65536, k_local=256, period=1024, S=4, mode=0),
    "C5": dict(N=16384, k_local=256, period=512, S=2, mode=0),
    "C6": dict(N=65536, k_local=256, period=1024, S=4, mode=2),
    "C7": dict(N=16384, k_local=256, period=512, S=2, mode=2),
}


def main():
    rec = {}
    for name, w in WORKLOADS.items():
        cnt, isum = oracle.counts(w["N"], w["k_local"], w["period"], w["S"], w["mode"])
        rec[name] = dict(w, pairs_per_head=int(cnt.sum()), index_sum_per_head=int(isum.sum()))
    doc = {
        "source": "written by tests/golden/make_golden.py from oracle.counts",
        "cite": "pi-Attention page, sections 2.1-2.2; ECP page, section 2 (PAR block)",
        "workloads": rec,
    }
    with open(os.path.join(HERE, "pair_counts.json"), "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
