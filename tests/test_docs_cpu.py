"""The documents name files that exist: every repository path quoted in README.md
(and every file a profile summary's command runs) is present, so the docs cannot drift from the
tree unnoticed."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "ragged_paged_attention_02_gb300"
EXTS = (".py", ".cu", ".cuh", ".h", ".c", ".md", ".txt", ".json")


def _quoted_paths(text):
    out = set()
    for tok in re.findall(r"`([^`\s]+)`", text):
        tok = tok.rstrip(".,;:)")
        if tok.startswith(("-", "$", "http")) or "(" in tok or "=" in tok:
            continue
        if tok.endswith(EXTS) or tok.endswith("/"):
            out.add(tok)
    return out


def _exists(path):
    # a bare file name may be quoted relative to the directory a table or paragraph is about
    for base in (ROOT, os.path.join(ROOT, PKG), os.path.join(ROOT, PKG, "csrc"), os.path.join(ROOT, "profiles"),
                 os.path.join(ROOT, "tests"), os.path.join(ROOT, "oracle"), os.path.join(ROOT, "include")):
        full = os.path.join(base, path)
        if glob.glob(full) or os.path.exists(full):
            return True
    return False


def test_paths_quoted_in_the_docs_exist():
    missing = []
    for doc in ("DESIGN.md", "README.md"):
        text = open(os.path.join(ROOT, doc)).read()
        for p in sorted(_quoted_paths(text)):
            if p in ("MEASURED_PEAKS.json", "librpa.so", "BASELINE.json", "PAPER.md"):
                continue  # written by others or built, not committed
            if not _exists(p):
                missing.append((doc, p))
    assert not missing, missing


def test_profile_commands_run_committed_files():
    for f in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(f).read()
        for script in re.findall(r"python ([\w/.]+\.py)", text):
            assert os.path.exists(os.path.join(ROOT, script)), (f, script)
        assert "_work" not in text, f
