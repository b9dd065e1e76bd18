"""Parsers for the hand-worked fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def read_cases(name: str) -> dict:
    """Read ``[case]`` sections of ``key = value`` lines; ``#`` starts a comment."""
    cases, cur = {}, None
    with open(os.path.join(HERE, name)) as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = line[1:-1]
                cases[cur] = {}
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            cases[cur][key] = val
    return cases
