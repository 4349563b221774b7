"""Reader for the text fixtures under tests/golden/ (values printed on the
source pages, each file headed by its citation)."""

import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    """Parse a fixture into {"layout": str, "grid": [[int]], key: [[int]]}.

    Lines starting with '#' are citations/comments.  A "grid" line starts a
    block of integer rows that runs until the next keyword line."""
    out: dict = {}
    grid = None
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for raw in fh:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            head, _, rest = line.partition(" ")
            if head == "layout":
                out["layout"] = rest.strip()
                grid = None
            elif head == "grid":
                grid = out.setdefault("grid", [])
            elif head.lstrip("-").isdigit() and grid is not None:
                grid.append([int(v) for v in line.split()])
            else:
                grid = None
                out.setdefault(head, []).append([int(v) for v in rest.split()])
    return out
