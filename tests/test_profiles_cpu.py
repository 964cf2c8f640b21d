"""The ncu summaries under profiles/ give the commands that made them.  Every
`python bench.py ...` command in them must parse with bench.py's own options
(so a summary never names a profile case, a dtype or a flag that no longer
exists), and every ncu command line in their code blocks must leave the GPU
clocks alone (`--clock-control none`)."""
import os
import re
import shlex
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _summaries():
    return sorted(n for n in os.listdir(PROFILES) if n.endswith((".md", ".txt")))


def _code_lines(text):
    """Lines of the fenced code blocks, backslash continuations joined."""
    out, in_block, cur = [], False, ""
    for line in text.splitlines():
        if line.strip().startswith("```"):
            in_block = not in_block
            continue
        if not in_block:
            continue
        if line.rstrip().endswith("\\"):
            cur += line.rstrip()[:-1] + " "
            continue
        out.append(cur + line)
        cur = ""
    return out


def _bench_commands():
    cases = []
    for name in _summaries():
        text = open(os.path.join(PROFILES, name)).read()
        for m in re.finditer(r"python bench\.py([^\n\"#`]*)", text):
            cases.append((name, m.group(1).strip()))
    return cases


def test_every_summary_names_its_command():
    names = _summaries()
    assert names, "no profile summaries"
    for name in names:
        text = open(os.path.join(PROFILES, name)).read()
        assert "python bench.py" in text, name
        assert re.search(r"\bncu\b", text), name


@pytest.mark.parametrize("name,args", _bench_commands())
def test_bench_command_parses(name, args):
    try:
        bench.build_parser().parse_args(shlex.split(args))
    except SystemExit as e:  # argparse reports an unknown option or choice by exiting
        pytest.fail(f"{name}: 'python bench.py {args}' does not parse ({e})")


@pytest.mark.parametrize("name", _summaries())
def test_ncu_commands_leave_the_clocks_alone(name):
    text = open(os.path.join(PROFILES, name)).read()
    for line in _code_lines(text):
        cmd = line.split("#", 1)[0]
        if re.match(r"\s*ncu\s+-", cmd) and not re.match(r"\s*ncu\s+-i\b", cmd):
            assert "--clock-control none" in cmd, f"{name}: {line.strip()}"
