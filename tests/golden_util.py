"""Reader for the `key = value  # citation` fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (t.strip() for t in line.split("=", 1))
            out[key] = int(val, 0) if val.lower().startswith("0x") else float(val)
    return out
