"""Parser for the hand-derived single-request traces in tests/golden/."""

from __future__ import annotations

import os
from typing import Dict, List, Tuple

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


RESIDENT = 1 << 30


def _val(x: str) -> int:
    """An integer; 'R<n>' is the resident row n (flagged)."""
    return RESIDENT | int(x[1:]) if x.startswith("R") else int(x)


def _ints(s: str) -> List[int]:
    return [_val(x) for x in s.split(",")] if s and s != "-" else []


def _kv(tokens: List[str]) -> Dict[str, str]:
    return dict(t.split("=", 1) for t in tokens)


def _checks(kv: Dict[str, str], op: dict) -> dict:
    """The optional status= (the op's own code, default 0) and word= (the
    request's status word after the op) of a prefill or backup line."""
    op["status"] = int(kv.get("status", 0))
    if "word" in kv:
        op["word"] = int(kv["word"])
    return op


def load(name: str) -> Tuple[Dict[str, int], List[Tuple[str, dict]]]:
    """Returns (layout {D,k,cap}, [(op, args)]), op in
    prefill/call/backup/resident/clear."""
    layout, ops = None, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            head, *rest = line.split()
            kv = _kv(rest)
            if head == "layout":
                layout = {k: int(v) for k, v in kv.items()}
            elif head == "prefill":
                ops.append(("prefill", _checks(kv, {"S": int(kv["S"])})))
            elif head == "call":
                ops.append(("call", {"S": int(kv["S"]), "topk": _ints(kv["topk"])}))
            elif head == "expect":
                plan = [] if kv["plan"] == "-" else \
                    [tuple(int(x) for x in p.split(":")) for p in kv["plan"].split(",")]
                ops[-1][1]["expect"] = {
                    "out": _ints(kv["out"]), "plan": plan, "status": int(kv["status"]),
                    "slot2tok": _ints(kv["slot2tok"]), "last_used": _ints(kv["last_used"])}
                if "word" in kv:
                    ops[-1][1]["expect"]["word"] = int(kv["word"])
            elif head == "backup":
                ops.append(("backup", _checks(kv, {"pos": int(kv["pos"])})))
            elif head == "clear":
                ops.append(("clear", {}))
            elif head == "resident":
                ops.append(("resident", {"ids": _ints(kv["ids"])}))
            else:
                raise ValueError(head)
    return layout, ops


def names() -> List[str]:
    return sorted(n for n in os.listdir(GOLDEN) if n.endswith(".txt"))
