"""Rules of the kernel sources that neither the compiler nor a GPU run can be
relied on to catch, checked on the CPU by reading the sources.

tcgen05.ld (tmem_load_32cols) leaves its destination registers undefined
until tcgen05.wait::ld (tmem_load_wait) has completed. The wait is a volatile
asm with a memory clobber: it keeps memory accesses after it, but not
arithmetic on the loaded registers, which the compiler may schedule above it
(an alpha * acc computed that early reads whatever the registers held before
the load landed). Every register array a TMEM load writes must therefore
pass through tmem_regs_ready, which reads and rewrites them, after the wait
and before anything else is loaded or waited for.
"""

import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "dense_fp32_gemm_major_gb300", "csrc")

_EVENT = re.compile(r"tmem_load_(?:16|32)cols\([^;]*?,\s*(?P<ld>\w+)\)\s*;"
                    r"|(?P<wait>tmem_load_wait\(\)\s*;)"
                    r"|tmem_regs_ready\((?P<ready>\w+)\)\s*;")


def _strip_comments(text: str) -> str:
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def fence_violations(text: str):
    """(line, message) for each TMEM load whose registers are not fenced after
    the wait that follows it."""
    text = _strip_comments(text)
    out = []
    loaded, waited = set(), set()
    for m in _EVENT.finditer(text):
        line = text.count("\n", 0, m.start()) + 1
        if m.group("ld"):
            if waited:
                out.append((line, f"load before {sorted(waited)} passed tmem_regs_ready"))
                waited = set()
            loaded.add(m.group("ld"))
        elif m.group("wait"):
            if waited:
                out.append((line, f"second wait before {sorted(waited)} passed tmem_regs_ready"))
            waited, loaded = set(loaded), set()
        else:
            name = m.group("ready")
            if name not in waited:
                out.append((line, f"tmem_regs_ready({name}) without a pending waited load"))
            waited.discard(name)
    if loaded:
        out.append((0, f"loads of {sorted(loaded)} never waited for"))
    if waited:
        out.append((0, f"{sorted(waited)} never passed tmem_regs_ready"))
    return out


def test_every_tmem_load_is_fenced_after_its_wait():
    checked = 0
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")) or name == "ptx.cuh":
            continue
        with open(os.path.join(CSRC, name)) as f:
            text = f.read()
        checked += len(re.findall(r"tmem_load_wait\(\)\s*;", text))
        bad = fence_violations(text)
        assert not bad, f"{name}: {bad}"
    assert checked >= 4  # the epilogue's four paths


def test_rule_catches_an_unfenced_use():
    # the rule itself, on made-up code: a wait with no fence, a fence of the
    # wrong array, and the correct form
    bad = """
      tmem_load_32cols(t, r0);
      tmem_load_32cols(t + 32, r1);
      tmem_load_wait();
      tmem_regs_ready(r0);
      float x = p.alpha * __uint_as_float(r1[0]);
    """
    assert fence_violations(bad), "missing fence of r1 not reported"
    wrong = """
      tmem_load_32cols(t, r);
      tmem_load_wait();
      tmem_regs_ready(q);
    """
    assert fence_violations(wrong)
    good = """
      tmem_load_32cols(t, r0);
      tmem_load_32cols(t + 32, r1);
      tmem_load_wait();
      tmem_regs_ready(r0);
      tmem_regs_ready(r1);
      tmem_load_32cols(t + 64, r0);
      tmem_load_wait();  // comment
      tmem_regs_ready(r0);
    """
    assert fence_violations(good) == []
