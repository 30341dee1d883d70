"""Reader for the page-number fixture (values printed on the pages)."""
import os

_HERE = os.path.dirname(os.path.abspath(__file__))


def _parse(v: str) -> float:
    v = v.strip()
    if v.startswith("2^"):
        return 2.0 ** float(v[2:])
    return float(v)


def page_numbers() -> dict:
    out = {}
    with open(os.path.join(_HERE, "page_numbers.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, value, _cite = (x.strip() for x in line.split("|", 2))
            out[name] = _parse(value)
    return out
