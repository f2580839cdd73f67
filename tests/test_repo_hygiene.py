"""Repository rules that a reader can check mechanically, on the CPU:

- no committed source, script or configuration file refers to a path inside
  the scratch folder at the repo root (scratch tools and experiments stay out
  of the product, and nothing committed may import, read or run them; review
  notes written about the repository are prose, not code, and are not
  checked);
- `profiles/` holds short text summaries only, each giving the full command
  that produced it, which runs a committed file (`bench.py`).

Skipped when the tree is not a git checkout.
"""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _tracked():
    try:
        out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True, timeout=60)
    except (OSError, subprocess.SubprocessError):
        pytest.skip("git is not available")
    if out.returncode != 0:
        pytest.skip("not a git checkout")
    return [f for f in out.stdout.splitlines() if f]


def test_nothing_committed_uses_the_scratch_folder():
    scratch = "_" + "work" + "/"  # spelled in parts so that this file does not match itself
    pattern = re.compile(r"(^|[^A-Za-z0-9_])" + re.escape(scratch))
    offenders = []
    code = (".py", ".cu", ".cuh", ".h", ".c", ".sh", ".ini", ".cfg", ".toml", ".json", ".txt")
    for f in _tracked():
        if f == ".gitignore" or not f.endswith(code) or re.match(r"[A-Z]+_r\d+\.json$", f):
            continue
        path = os.path.join(ROOT, f)
        try:
            text = open(path, encoding="utf-8").read()
        except (UnicodeDecodeError, OSError):
            continue
        if pattern.search(text):
            offenders.append(f)
    assert offenders == []


def test_profiles_are_text_summaries_with_their_command():
    files = [f for f in _tracked() if f.startswith("profiles/")]
    assert files, "no committed profile summaries"
    for f in files:
        assert f.endswith((".md", ".txt")), f
        path = os.path.join(ROOT, f)
        assert os.path.getsize(path) < 16 * 1024, f
        text = open(path, encoding="utf-8").read()
        # the command runs committed files: the benchmark or the package's tools
        assert "Command" in text, f
        assert "python bench.py" in text or "python -m mamba_chunked_ssd_gb300." in text, f
        assert "--clock-control none" in text, f
