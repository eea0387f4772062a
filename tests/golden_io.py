"""Reader for the hand-derived golden stream fixtures in tests/golden/."""
from __future__ import annotations

from pathlib import Path

import numpy as np

GOLDEN = Path(__file__).resolve().parent / "golden"


def parse_input(spec: str) -> bytes:
    parts = spec.split()
    kind, items = parts[0], parts[1:]
    if kind == "hex":
        return bytes(int(x, 16) for x in items)
    dt = {"u32": "<u4", "u16": "<u2"}[kind]
    vals = []
    for it in items:
        v, n = it.split("*")
        vals += [int(v, 0)] * int(n)
    return np.array(vals, dtype=dt).tobytes()


def load(path: Path) -> dict:
    rec = {"name": path.stem}
    for line in path.read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(" ")
        if key == "elem_width":
            rec["elem_width"] = int(val)
        elif key == "input":
            rec["input"] = parse_input(val)
        elif key == "stream":
            rec["stream"] = bytes(int(x, 16) for x in val.split())
    return rec


def all_cases() -> list[dict]:
    return [load(p) for p in sorted(GOLDEN.glob("*.txt"))]
