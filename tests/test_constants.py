"""The defaults of the oracle and of the input generator are the constants the pages print."""
import json
import os

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")


def page_constants():
    with open(GOLDEN) as f:
        d = json.load(f)
    return {k: v["value"] for k, v in d.items() if not k.startswith("_")}


def test_oracle_defaults_are_the_pages_constants():
    assert oracle.DEFAULT_CONFIG == page_constants()


def test_generator_defaults_are_the_pages_constants():
    assert workloads.DEFAULT_CONFIG == page_constants()
