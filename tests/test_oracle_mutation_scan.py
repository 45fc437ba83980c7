"""Mechanical mutation scan of the oracle against its pins.

Every code line of the oracle is edited one way at a time: a `+` or `-`
swapped, an integer literal moved by one, a comparison loosened or flipped,
max/min or rint/floor swapped, `&` turned into `|`, an `abs` dropped.  Each
edited copy runs the pins (test_oracle_encodings.py, test_oracle_path.py);
an edit that no pin catches must appear in EQUIVALENT below with the reason
it cannot change a result on the oracle's domain (finite fp32 activations,
E4M3 codes, E8M0 bytes, fp32 scales, D % 16 == 0).  A change to the oracle
that opens a real gap therefore fails this test until a pin covers it.
"""

import re

from pins_harness import failing_pins, oracle_from_source, oracle_source

_SWAPS = ((">=", ">"), ("<=", "<"), (" > ", " >= "), (" < ", " <= "), ("==", "!="),
          ("np.max", "np.min"), ("np.maximum", "np.minimum"), ("np.rint", "np.floor"),
          ("&", "|"), ("np.abs(", "("))

# (line, edited line) -> why the edit cannot change any result on the domain
EQUIVALENT = {
    ("E4M3_MAX = 448.0", "E4M3_MAX = 449.0"):
        "only used by the explicit saturation line, which the clipped nearest-value search already implies",
    ("E4M3_MAX = 448.0", "E4M3_MAX = 447.0"):
        "values in [447, 448) round to 448 (0x7E) anyway: the midpoint below 448 is 432",
    ("E4M3_MAX = 448.0", "E4M3_MAX = 448.1"):
        "the clipped search maps everything above 448 to 0x7E anyway",
    ("hi = np.clip(hi, 0, 0x7E)", "hi = np.clip(hi, 1, 0x7E)"):
        "hi = 0 only for a = 0, where lo = 0 is picked (distance 0) either way",
    ("code = np.where(a >= E4M3_MAX, 0x7E, code)", "code = np.where(a > E4M3_MAX, 0x7E, code)"):
        "a == 448 is found exactly by the search (code 0x7E)",
    ("e = np.where(amax == 0.0, -127, e)", "e = np.where(amax == 0.0, -128, e)"):
        "the clamp to [-127, 127] on the next line restores -127",
    ("if R == 0:", "if R == 1:"):
        "with R == 0 the general path moves no element (empty slices); R is even",
    ("KG = (D + GROUP - 1) // GROUP", "KG = (D + GROUP - 2) // GROUP"):
        "differs only when D % 128 == 1, and D % 16 == 0",
    ("a = np.abs(v)", "a = (v)"):
        "bf16 rounding: rint is symmetric, the float32 conversion carries the sign and overflows to -inf",
    ("r = np.where(a == 0.0, 0.0, r)", "r = np.where(a == 0.1, 0.0, r)"):
        "a zero input already gives r = 0 (frexp(0) = (0, 0), rint(0) = 0)",
    ("r = np.where(r >= 2.0 ** 128, np.inf, r)", "r = np.where(r >= 3.0 ** 128, np.inf, r)"):
        "the float32 conversion turns any r >= 2^128 into inf anyway",
    ("r = np.where(r >= 2.0 ** 128, np.inf, r)", "r = np.where(r >= 2.1 ** 128, np.inf, r)"):
        "the float32 conversion turns any r >= 2^128 into inf anyway",
    ("r = np.where(r >= 2.0 ** 128, np.inf, r)", "r = np.where(r >= 2.0 ** 129, np.inf, r)"):
        "the float32 conversion turns any r >= 2^128 into inf anyway",
    ("r = np.where(r >= 2.0 ** 128, np.inf, r)", "r = np.where(r > 2.0 ** 128, np.inf, r)"):
        "the float32 conversion turns r == 2^128 into inf anyway",
    ("a = np.abs(np.asarray(y_ref, dtype=np.float64))", "a = (np.asarray(y_ref, dtype=np.float64))"):
        "bf16_ulp uses only the frexp exponent, which is the same for y and -y",
    ("ok = np.isfinite(s) & (s > 0) & (m == 0.5) & (k >= -127) & (k <= 127)",
     "ok = np.isfinite(s) & (s > 0) & (m == 0.5) & (k >= -127) & (k <= 128)"):
        "the input is float32, whose largest power of two is 2^127",
    ("ok = np.isfinite(s) & (s > 0) & (m == 0.5) & (k >= -127) & (k <= 127)",
     "ok = np.isfinite(s) & (s >= 0) & (m == 0.5) & (k >= -127) & (k <= 127)"):
        "zero fails m == 0.5 (frexp(0) gives m = 0)",
}


def _code_lines(src):
    """(index, code part) of every line outside docstrings, comments, defs and imports."""
    in_doc = False
    for i, ln in enumerate(src.split("\n")):
        st = ln.strip()
        if '"""' in st:
            if st.count('"""') == 1:
                in_doc = not in_doc
            continue
        if in_doc or not st or st.startswith(("#", "def ", "import ", "from ")):
            continue
        yield i, ln.split("#")[0]


def _edits(code):
    for m in re.finditer(r"(?<![=<>!*])([+\-])(?![=*])", code):
        if m.start() > 1 and code[m.start() - 1] in "eE" and code[m.start() - 2].isdigit():
            continue  # exponent of a float literal
        yield code[:m.start()] + ("-" if m.group(1) == "+" else "+") + code[m.end():]
    for m in re.finditer(r"\b(\d+)\b", code):
        v = int(m.group(1))
        for nv in (v + 1, v - 1):
            if nv >= 0:
                yield code[:m.start()] + str(nv) + code[m.end():]
    for a, b in _SWAPS:
        j = code.find(a)
        while j >= 0:
            yield code[:j] + b + code[j + len(a):]
            j = code.find(a, j + 1)


def test_every_uncaught_edit_is_an_equivalent_one():
    src = oracle_source()
    lines = src.split("\n")
    tried, survivors = 0, []
    for i, code in _code_lines(src):
        for edited in _edits(code):
            if edited == code:
                continue
            new = list(lines)
            new[i] = edited + lines[i][len(code):]
            try:
                mod = oracle_from_source("\n".join(new))
            except Exception:
                continue  # the edit does not even compile or import
            tried += 1
            if not failing_pins(mod, stop_at_first=True):
                survivors.append((code.strip(), edited.strip()))
    assert tried > 200
    unexplained = [s for s in survivors if s not in EQUIVALENT]
    assert not unexplained, "edits no pin catches: " + "; ".join(f"{a!r} -> {b!r}" for a, b in unexplained)
