"""Loads the cited fixtures under tests/golden/."""
import json
import os

_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str):
    with open(os.path.join(_DIR, name)) as f:
        return json.load(f)
