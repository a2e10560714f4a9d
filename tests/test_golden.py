"""Values the source pages print for a worked example (fixtures under
tests/golden/, each naming its passage), checked against our reading of the
formulas they come from."""
import json
import math
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_issue261_static_traffic_model_example():
    """Issue #261 prints, for N=4096, D=2048, V=32768: default chunking gives
    K = 8, and the proposed accumulation saves 4.0 GiB of gradient-table
    traffic.  Our reading: C = floor(2^24 / V) rows per chunk, K = ceil(N / C),
    saving = 8 K V D bytes, GiB = 2^30 bytes."""
    g = _load("issue261_static_traffic_model.json")
    N, D, V = g["example"]["N"], g["example"]["D"], g["example"]["V"]
    C = (1 << 24) // V
    K = math.ceil(N / C)
    assert K == g["printed"]["K"]
    saving = 8 * K * V * D
    assert round(saving / 2 ** 30, 1) == g["printed"]["saving_GiB"]
    current = 4 * V * D + 16 * K * V * D
    candidate = 4 * V * D + 8 * K * V * D
    assert current - candidate == saving

