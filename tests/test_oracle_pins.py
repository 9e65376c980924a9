"""The FP64 oracle against its pins (CPU only), and the pins against planted
mistakes: every deliberately mutated oracle build must fail at least one pin."""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    fails = pin(oracle_lib)
    assert not fails, "\n".join(fails[:10])


# mutation -> what it plants (see ORACLE_MUTATION in oracle/paged_attn_oracle.c)
MUTATIONS = {
    1: "drops the 1/sqrt(D) softmax scale",
    2: "causal window one key short",
    3: "query head -> KV head as h % Hkv",
    4: "E4M3 exponent bias 8",
    5: "V scale not applied",
    6: "page and slot index swapped",
    7: "exp(max - s) sign error",
    8: "E4M3 subnormals decoded as normals",
    9: "FP16 exponent bias 16",
    10: "lse without the max term",
    11: "E5M2 exponent bias 16",
    12: "E5M2 subnormals decoded as normals",
    13: "selected row written to the slot of its row index instead of its list position",
    14: "one score / accumulator scratch shared by every thread",
}


_CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
lib = oracle.load(mutation={mutation}, out_dir={out_dir!r})
assert lib.oracle_mutation() == {mutation}
for pin in oracle_pins.ALL_PINS:
    try:
        fails = pin(lib)
    except Exception as e:
        fails = [repr(e)]
    print(pin.__name__, "FAIL" if fails else "pass", flush=True)
"""


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_pins_catch_mutation(mutation, tmp_path_factory):
    """Each mutant runs in a child process: a planted indexing mistake may read
    out of bounds and crash, which also counts as caught."""
    out_dir = str(tmp_path_factory.mktemp(f"mut{mutation}"))
    oracle.build(mutation=mutation, out_dir=out_dir)
    here = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(here), tests=here, mutation=mutation, out_dir=out_dir)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    lines = [ln.split() for ln in r.stdout.splitlines() if ln.strip()]
    caught = [ln[0] for ln in lines if len(ln) == 2 and ln[1] == "FAIL"]
    crashed = r.returncode != 0
    assert caught or crashed, f"mutation {mutation} ({MUTATIONS[mutation]}) passed every pin:\n{r.stdout}{r.stderr}"
