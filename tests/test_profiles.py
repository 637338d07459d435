"""The committed profile summaries cite commands that can be rerun from the repository.

Every ncu capture named in `profiles/*.md` leaves the GPU clocks alone
(`--clock-control none`), and every program a summary runs is a committed file of the
repository (no scratch scripts).
"""

import os
import re

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
PROFILES = os.path.join(ROOT, "profiles")
FILES = sorted(f for f in os.listdir(PROFILES) if f.endswith((".md", ".txt")))


def _commands(text: str):
    """Shell commands in the summary's code blocks, continuation lines joined."""
    out = []
    for block in re.findall(r"```[^\n]*\n(.*?)```", text, flags=re.S):
        joined = re.sub(r"\\\n\s*", " ", block)
        out += [ln.strip() for ln in joined.splitlines() if ln.strip() and
                not ln.strip().startswith("#")]
    return out


def test_there_are_profiles():
    assert FILES


@pytest.mark.parametrize("name", FILES)
def test_ncu_captures_leave_clocks_alone(name):
    text = open(os.path.join(PROFILES, name)).read()
    for cmd in _commands(text):
        for part in cmd.split("&&"):
            part = part.strip()
            if part.startswith("ncu ") and not re.search(r"\s-i\s", part):
                assert "--clock-control none" in part, (name, part)


@pytest.mark.parametrize("name", FILES)
def test_programs_are_committed_files(name):
    text = open(os.path.join(PROFILES, name)).read()
    for cmd in _commands(text):
        for script in re.findall(r"\bpython3?\s+([\w./-]+\.py)", cmd):
            path = os.path.normpath(os.path.join(ROOT, script))
            assert os.path.isfile(path), (name, script)
            assert "_work" not in script.split(os.sep), (name, script)
