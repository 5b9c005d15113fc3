"""Static checks of the CUDA sources (no GPU): every spin-wait is bounded, nothing
traps, every tiled TMA copy starts on a 16-byte boundary, and the tensor-core MMAs
never mix operand types.

Each kernel's mbarrier waits go through one helper, ``mbar_wait``, which polls
``mbarrier.try_wait`` and gives up after a %globaltimer limit (setting the kernel's
abort flag), so a lost arrival ends the kernel with KVC_DEV_TIMEOUT instead of hanging
the GPU.  These tests keep it that way: a loop without an exit condition must sit in
such a helper, ``try_wait`` may be polled nowhere else, and no device code traps or
asserts.
"""
import glob
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "diffusion_serving_gb300", "csrc")
SOURCES = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.h")))


def code(path):
    """The source without // and /* */ comments."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def block_from(text, start):
    """From `start` to the brace that closes the first `{` after it."""
    i = text.index("{", start) + 1
    depth = 1
    while depth:
        depth += {"{": 1, "}": -1}.get(text[i], 0)
        i += 1
    return text[start:i]


def function_bodies(text, name):
    """Definitions of the bool-returning device helpers called `name`."""
    return [block_from(text, m.start()) for m in re.finditer(r"\bbool\s+%s\s*\(" % re.escape(name), text)]


def test_sources_found():
    names = {os.path.basename(p) for p in SOURCES}
    assert {"k_attn_tc.cu", "k_decode.cu", "k_cache.cu", "kvc_api.cu"} <= names


def test_unconditional_loops_are_bounded_waits():
    """A loop without an exit condition is either mbar_wait's polling loop (which has a
    time limit) or a work loop that leaves with `break` (each of its waits a bounded
    mbar_wait, checked below); there are no while / do loops to poll a flag with."""
    for path in SOURCES:
        text = code(path)
        name = os.path.basename(path)
        assert not re.search(r"\bwhile\s*\(", text) and not re.search(r"\bdo\s*\{", text), \
            f"{name}: a while / do loop (polling loops go through mbar_wait)"
        bodies = function_bodies(text, "mbar_wait")
        for m in re.finditer(r"\bfor\s*\([^;)]*;\s*;", text):
            if any(text.find(b) <= m.start() < text.find(b) + len(b) for b in bodies):
                continue
            assert "break;" in block_from(text, m.start()), f"{name}: a loop without an exit condition or break"
        for b in bodies:
            assert "globaltimer()" in b and "kTimeoutNs" in b and "return false" in b, \
                f"{os.path.basename(path)}: mbar_wait without a time limit"


def test_try_wait_is_polled_only_by_the_bounded_helper():
    for path in SOURCES:
        text = code(path)
        bodies = function_bodies(text, "mbar_wait")
        stripped = text
        for b in bodies:
            stripped = stripped.replace(b, "")
        defs = function_bodies(stripped, "mbar_try_wait")
        for d in defs:
            stripped = stripped.replace(d, "")
        assert "mbar_try_wait(" not in stripped, f"{os.path.basename(path)}: try_wait polled outside mbar_wait"
        assert "mbarrier.try_wait" not in stripped, f"{os.path.basename(path)}: raw try_wait outside the helpers"


def test_timeouts_are_short():
    for path in SOURCES:
        for m in re.finditer(r"kTimeoutNs\s*=\s*(\d+)ull", code(path)):
            assert int(m.group(1)) <= 2_000_000_000, f"{os.path.basename(path)}: wait limit above 2 s"


def test_no_device_traps_or_asserts():
    for path in SOURCES:
        text = code(path)
        assert "__trap" not in text and not re.search(r"\btrap\s*;", text), os.path.basename(path)
        assert not re.search(r"(?<!static_)\bassert\s*\(", text), os.path.basename(path)
        assert "__brkpt" not in text, os.path.basename(path)


def call_args(text, start):
    """Arguments of the call whose '(' follows `start`, split at depth-0 commas."""
    i = text.index("(", start) + 1
    depth, cur, args = 1, "", []
    while True:
        ch = text[i]
        if ch in "([{":
            depth += 1
        elif ch in ")]}":
            depth -= 1
            if depth == 0:
                args.append(cur.strip())
                return args
        if ch == "," and depth == 1:
            args.append(cur.strip())
            cur = ""
        else:
            cur += ch
        i += 1


def test_tma_inner_coordinate_is_16_byte_aligned():
    """A tiled cp.async.bulk.tensor copy must start at an innermost coordinate whose byte
    offset is a multiple of 16: nothing checks it before the copy runs, and a misaligned
    one stops the context.  Every tensor map is over 16-bit elements (kvc_make_tile_map
    refuses other types), so x must be a multiple of 8 elements: each call site's x is a
    multiple of a literal, and that literal a multiple of 8."""
    api = code(os.path.join(CSRC, "kvc_api.cu"))
    make = block_from(api, api.index("bool kvc_make_tile_map("))
    assert "dtype != KVC_BF16 && dtype != KVC_F16" in make and "return false" in make
    sites = 0
    for path in SOURCES:
        text = code(path)
        for name, x_index in (("tma_load_4d", 3), ("tma_store_4d", 2)):
            for m in re.finditer(r"\b%s\s*\(" % name, text):
                if re.search(r"void\s+$", text[max(0, m.start() - 40):m.start()]):
                    continue                                   # the definition
                x = call_args(text, m.start())[x_index]
                lit = re.fullmatch(r"(?:\w+\s*\*\s*(\d+)|(\d+)\s*\*\s*\w+|(\d+))", x)
                assert lit, f"{os.path.basename(path)}: TMA x coordinate '{x}' is not literal-aligned"
                assert int(next(g for g in lit.groups() if g)) % 8 == 0, f"{os.path.basename(path)}: x = {x}"
                sites += 1
    assert sites >= 8


def test_mma_operands_share_one_type():
    """In one tcgen05.mma of kind::f16, A and B must have the same type.  The instruction
    descriptor takes a single format for both (bits 7-9 for A, 10-12 for B), every
    descriptor of a kernel is built from the kernel's element type, and P, the A operand
    of the PV MMA read from TMEM, is packed in that same type."""
    text = code(os.path.join(CSRC, "k_attn_tc.cu"))
    body = block_from(text, text.index("constexpr uint32_t idesc_f16("))
    assert re.search(r"\(fmt << 7\) \| \(fmt << 10\)", body), body
    calls = re.findall(r"idesc_f16\(([^,]+),", text)
    calls = [c.strip() for c in calls if not c.strip().startswith("uint32_t")]
    assert calls and all(c == "kBf16 ? 1u : 0u" for c in calls), calls
    packs = re.findall(r"pack2<(\w+)>", text)
    assert packs and all(t == "kBf16" for t in packs), packs
    assert "kind::f16" in text and "kind::tf32" not in text and "kind::f8f6f4" not in text

