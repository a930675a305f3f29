"""The tile-override grammar (qg_set_tile_override / QGEMV_TILE), CPU: random specs
are accepted exactly when a plain model of the grammar accepts them."""
from __future__ import annotations

import random

import block_quantized_token_format_gb300 as qg

# key -> allowed integer values (the instantiated kernels and the documented ranges)
ALLOWED = {
    "rpw": {1, 2, 3, 4, 5, 6, 8},
    "depth": set(range(2, 17)),
    "warps": set(range(1, 17)),
    "ctas": set(range(1, 9)),
    "pre": set(range(1, 17)),
    "split": set(range(1, 9)),
    "gw": set(range(0, 65)),
}


def model_accepts(spec: str) -> bool:
    for item in spec.split(","):
        if item == "":
            continue
        if item.count("=") != 1:
            return False
        key, val = item.split("=")
        if key not in ALLOWED or not val.isdigit() or not (1 <= len(val) <= 3):
            return False
        if int(val) not in ALLOWED[key]:
            return False
    return True


def random_spec(rng: random.Random) -> str:
    items = []
    for _ in range(rng.randint(0, 4)):
        key = rng.choice(list(ALLOWED) + ["foo", "rp", "RPW", ""])
        val = rng.choice([str(rng.randint(0, 20)), str(rng.randint(0, 99)), "-1", "x", "", "0007", "1e1"])
        items.append(rng.choice([f"{key}={val}", f"{key}{val}", f"{key}=={val}"]) if rng.random() < 0.1
                     else f"{key}={val}")
    return ",".join(items) + ("," if rng.random() < 0.1 else "")


def test_random_specs_match_the_grammar_model():
    lib = qg.load_library()
    rng = random.Random(1234)
    n_ok = 0
    try:
        for _ in range(3000):
            spec = random_spec(rng)
            want = model_accepts(spec)
            got = lib.qg_set_tile_override(spec.encode()) == 0
            assert got == want, spec
            n_ok += want
    finally:
        lib.qg_set_tile_override(None)
    assert n_ok > 100                      # the generator reaches both sides of the grammar
