"""Reader for tests/golden/*.ini: the worked examples printed on the pages."""
import configparser
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str = "worked_examples.ini") -> dict:
    cp = configparser.ConfigParser(interpolation=None)
    cp.read(os.path.join(GOLDEN, name))
    out = {}
    for sec in cp.sections():
        d = {}
        for k, v in cp.items(sec):
            if k in ("source", "op", "predicate"):
                d[k] = v
            elif k in ("total", "count"):
                d[k] = int(v)
            else:
                d[k] = [float(t) if "." in t else int(t) for t in v.split()]
        out[sec] = d
    return out
