"""Summarise a parity log written by the GPU tests (test infrastructure).

    SV_PARITY_LOG=gpurun_out/parity.jsonl python -m pytest tests -m gpu -q
    python tests/parity_summary.py gpurun_out/parity.jsonl

Prints one markdown row per case family (the label without its seed or call
number): the sequences compared with the oracle, the near-ties split into
accept-test ties and draw ties, the disagreements inside the bands, the
disagreements outside them (always 0 in a passing run), and the largest
difference between the kernel's and the oracle's distances from the draw
target to the chosen token's interval edges.
"""
from __future__ import annotations

import collections
import json
import sys


def family(label: str) -> str:
    for cut in (" seed", " call"):
        label = label.split(cut)[0]
    return label


def summarise(lines):
    agg = collections.OrderedDict()
    for line in lines:
        r = json.loads(line)
        a = agg.setdefault(family(r["case"]), collections.Counter())
        a["calls"] += 1
        a["sequences"] += r["sequences"]
        a["accept"] += r.get("accept_near_ties", 0)
        a["draw"] += r.get("draw_near_ties", r["near_ties"] - r.get("accept_near_ties", 0))
        a["tie_mismatches"] += r["near_tie_mismatches"]
        a["mismatches"] += r["mismatches"]
        a["edge_seqs"] += r.get("draw_edge_seqs", 0)
        a["edge_err"] = max(a["edge_err"], r.get("draw_edge_err", 0.0))
    return agg


def main(path: str) -> None:
    with open(path) as f:
        agg = summarise(f)
    print("| case | calls | sequences | accept ties | draw ties | ties % | disagreements in ties "
          "| outside ties | draw-edge error (max, sequences) |")
    print("|---|---|---|---|---|---|---|---|---|")
    tot = collections.Counter()
    for k, a in agg.items():
        pct = 100.0 * (a["accept"] + a["draw"]) / max(1, a["sequences"])
        err = f"{a['edge_err']:.2e} ({a['edge_seqs']})" if a["edge_seqs"] else "-"
        print(f"| {k} | {a['calls']} | {a['sequences']} | {a['accept']} | {a['draw']} | {pct:.2f} "
              f"| {a['tie_mismatches']} | {a['mismatches']} | {err} |")
        for key in ("sequences", "accept", "draw", "tie_mismatches", "mismatches", "edge_seqs"):
            tot[key] += a[key]
        tot["edge_err"] = max(tot["edge_err"], a["edge_err"])
    pct = 100.0 * (tot["accept"] + tot["draw"]) / max(1, tot["sequences"])
    print(f"| all | | {tot['sequences']} | {tot['accept']} | {tot['draw']} | {pct:.2f} "
          f"| {tot['tie_mismatches']} | {tot['mismatches']} | {tot['edge_err']:.2e} ({tot['edge_seqs']}) |")


if __name__ == "__main__":
    main(sys.argv[1])
