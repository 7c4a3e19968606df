"""CPU-only checks of the library boundary: it loads, exports every symbol the
public header declares, and its host logic (size helpers, split plan, status
strings, argument validation that returns before any launch) behaves."""
import ctypes
import os
import re

import pytest

import paged_kv_gqa_10_gb300 as pgqa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgqa.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pgqa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pgqa_kv_cache_write", "pgqa_paged_attention_decode", "pgqa_paged_prefill_varlen",
              "pgqa_paged_kv_gather", "pgqa_decode_workspace_size", "pgqa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(pgqa.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version_and_status_strings():
    assert pgqa.abi_version() == pgqa.ABI_VERSION
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert pgqa.status_string(code) and pgqa.status_string(code) != "unknown status"
    assert pgqa.status_string(-99) == "unknown status"


def test_kv_cache_bytes_matches_printed_figures():
    with open(os.path.join(GOLDEN, "kv_cache_size.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for layers, tokens, heads, dim, elem, printed, tol in rows:
        dt = pgqa.BF16 if int(elem) == 2 else pgqa.E4M3
        got = pgqa.kv_cache_bytes(int(layers), int(tokens), int(heads), int(dim), dt) / 1e9
        assert abs(got - float(printed)) <= float(tol), (got, printed)
    assert pgqa.kv_cache_bytes(1, 16, 1, 128, pgqa.BF16) == 8192  # one 16-token K+V page
    assert pgqa.kv_cache_bytes(1, 16, 1, 128, pgqa.E4M3) == 4096
    assert pgqa.kv_cache_bytes(-1, 1, 1, 1) == -1


@pytest.mark.parametrize("sms", [1, 148, 152])
@pytest.mark.parametrize("D,dt", [(128, pgqa.BF16), (64, pgqa.BF16), (128, pgqa.E4M3)])
def test_decode_grid_fills_every_sm(sms, D, dt):
    g = pgqa.decode_grid_size(sms, D, dt)
    assert g >= sms and g % sms == 0          # the same number of CTAs on every SM


def test_decode_grid_rejects_bad_arguments():
    for args in ((0, 128, pgqa.BF16), (152, 96, pgqa.BF16), (152, 128, 9)):
        with pytest.raises(pgqa.PgqaError):
            pgqa.decode_grid_size(*args)


def _call_decode(**over):
    a = dict(out=1 << 20, lse=None, q=1 << 20, k=1 << 20, v=1 << 20, bt=1 << 20, maxb=4,
             cl=1 << 20, B=2, Hq=8, Hkv=2, D=128, NB=16, bs=16, scale=0.1, dtype=0, ks=None,
             vs=None, maxctx=64, ws=None, wsb=0, st=None)
    a.update(over)
    f = pgqa.lib.pgqa_paged_attention_decode
    return f(a["out"], a["lse"], a["q"], a["k"], a["v"], a["bt"], a["maxb"], a["cl"], a["B"],
             a["Hq"], a["Hkv"], a["D"], a["NB"], a["bs"], a["scale"], a["dtype"], a["ks"], a["vs"],
             a["maxctx"], a["ws"], a["wsb"], a["st"], None)


@pytest.mark.parametrize("over,want", [
    (dict(Hq=7), pgqa.EINVAL),                 # heads not a multiple of kv heads
    (dict(Hq=32, Hkv=2), pgqa.EUNSUPPORTED),   # group of 16
    (dict(D=96), pgqa.EUNSUPPORTED),
    (dict(bs=64), pgqa.EUNSUPPORTED),          # decode reads 8-, 16- and 32-token blocks
    (dict(bs=4), pgqa.EUNSUPPORTED),
    (dict(bs=32, NB=1 << 25), pgqa.EUNSUPPORTED),  # cache rows past int32
    (dict(dtype=7), pgqa.EUNSUPPORTED),
    (dict(dtype=1), pgqa.EINVAL),              # E4M3 without scales
    (dict(dtype=1, D=96, ks=1 << 20, vs=1 << 20), pgqa.EUNSUPPORTED),  # E4M3 at head_dim 96
    (dict(ks=1 << 20, vs=1 << 20), pgqa.EINVAL),  # scales given for bf16
    (dict(B=-1), pgqa.EINVAL),
    (dict(scale=float("nan")), pgqa.EINVAL),
    (dict(q=None), pgqa.EINVAL),
    (dict(q=(1 << 20) + 8), pgqa.EINVAL),      # misaligned
    (dict(B=0), pgqa.OK),                      # nothing to do, nothing launched
])
def test_decode_argument_validation(over, want):
    assert _call_decode(**over) == want


def test_kv_write_argument_validation():
    f = pgqa.lib.pgqa_kv_cache_write
    P = 1 << 20
    assert f(P, P, P, 4, 2, 100, P, P, 8, 16, 0, None, None, None, None) == pgqa.EUNSUPPORTED
    assert f(P, P, P, 4, 2, 128, P, P, 8, 16, 1, None, None, None, None) == pgqa.EINVAL
    assert f(P, P, P, 0, 2, 128, P, P, 8, 16, 0, None, None, None, None) == pgqa.OK
    assert f(None, P, P, 4, 2, 128, P, P, 8, 16, 0, None, None, None, None) == pgqa.EINVAL


def test_prefill_argument_validation():
    f = pgqa.lib.pgqa_paged_prefill_varlen
    P = 1 << 20
    #       out lse q  T    k  v  bt maxb cu S  maxL Hq Hkv D    NB  bs  scale ws  wsb st  stream
    args = [P, None, P, 100, P, P, P, 4, P, 2, 64, 8, 2, 128, 16, 16, 0.1, None, 0, None, None]
    assert f(*args[:13], 96, *args[14:]) == pgqa.EUNSUPPORTED
    assert f(*args[:11], 7, *args[12:]) == pgqa.EINVAL
    assert f(*args[:9], 0, *args[10:]) == pgqa.OK
    assert f(*args[:3], -1, *args[4:]) == pgqa.EINVAL
    assert f(*args[:16], -0.1, *args[17:]) == pgqa.EINVAL          # scale must be > 0
    assert f(*args[:9], 5000, *args[10:]) == pgqa.EUNSUPPORTED     # more than 4096 sequences
    assert f(*args) == pgqa.ENOWORKSPACE                           # no workspace given
    assert f(*args[:10], 600000, *args[11:]) == pgqa.EUNSUPPORTED  # longer than 524288 tokens
    assert pgqa.prefill_workspace_size(2, 8, 64) == 256 + (4096 + 2 * 2048) * 4


def test_prefill_kv_argument_validation():
    f = pgqa.lib.pgqa_paged_prefill_varlen_kv
    P = 1 << 20
    #       out lse q  T    k  v  bt maxb cuq lk S  maxq maxk Hq Hkv D   NB  bs  scale ws wsb st stream
    args = [P, None, P, 100, P, P, P, 64, P, P, 2, 64, 1000, 8, 2, 128, 64, 16, 0.1, P, 33024, None,
            None]
    assert f(*args[:9], None, *args[10:]) == pgqa.EINVAL           # no key lengths
    assert f(*args[:12], 1 << 27, *args[13:]) == pgqa.EUNSUPPORTED  # keys beyond 2^26
    assert f(*args[:12], -1, *args[13:]) == pgqa.EINVAL
    assert f(*args[:10], 0, *args[11:]) == pgqa.OK                 # nothing to do
    assert f(*args[:19], None, 0, *args[21:]) == pgqa.ENOWORKSPACE


def test_prefill_e4m3_argument_validation():
    f = pgqa.lib.pgqa_paged_prefill_varlen_e4m3
    P = 1 << 20
    #       out lse q  T    k  v  bt maxb cuq lk    S  maxq maxk Hq Hkv D   NB  bs  scale ks vs
    args = [P, None, P, 100, P, P, P, 64, P, None, 2, 64, 0, 8, 2, 128, 64, 16, 0.1, P, P,
            P, 33024, None, None]  # ws wsb st stream
    assert f(*args[:19], None, *args[20:]) == pgqa.EINVAL          # no k_scale
    assert f(*args[:20], None, *args[21:]) == pgqa.EINVAL          # no v_scale
    assert f(*args[:19], P + 2, *args[20:]) == pgqa.EINVAL         # misaligned scales
    assert f(*args[:15], 96, *args[16:]) == pgqa.EUNSUPPORTED      # head_dim 96
    assert f(*args[:17], 32, *args[18:]) == pgqa.EUNSUPPORTED      # 32-token blocks
    assert f(*args[:10], 0, *args[11:]) == pgqa.OK                 # nothing to do
    assert f(*args[:21], None, 0, *args[23:]) == pgqa.ENOWORKSPACE


def test_decode_append_argument_validation():
    f = pgqa.lib.pgqa_paged_attention_decode_append
    P = 1 << 20
    #       out lse q  key val k  v  bt maxb cl B  Hq Hkv D    NB  bs  scale dt ks    vs
    args = [P, None, P, P, P, P, P, P, 4, P, 2, 8, 2, 128, 16, 16, 0.1, 0, None, None,
            64, None, 0, None, None]  # maxctx ws wsb st stream
    assert f(*args[:3], None, *args[4:]) == pgqa.EINVAL            # no new K rows
    assert f(*args[:4], None, *args[5:]) == pgqa.EINVAL            # no new V rows
    assert f(*args[:3], P + 8, *args[4:]) == pgqa.EINVAL           # misaligned rows
    assert f(*args[:15], 64, *args[16:]) == pgqa.EUNSUPPORTED      # 64-token blocks
    assert f(*args[:10], 0, *args[11:]) == pgqa.OK                 # nothing to do


def test_binding_signatures_match_the_header():
    """Every function the binding declares takes as many arguments as the header says."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decl = {m.group(1): m.group(2) for m in
            re.finditer(r"\b(pgqa_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text)}
    lib = pgqa._handle()
    checked = 0
    for name, params in decl.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        checked += 1
    assert checked >= 12


def test_every_entry_point_has_a_python_binding():
    """Each function the header declares is reachable from Python under the same name
    without the ``pgqa_`` prefix, and is listed in the package's ``__all__``."""
    for name in declared_functions():
        short = name[len("pgqa_"):]
        assert callable(getattr(pgqa, short, None)), short
        assert short in pgqa.__all__, short


def test_wait_limit_setter_rejects_negative_and_restores_default():
    with pytest.raises(ValueError):
        pgqa.set_decode_wait_limit_ns(-1)
    pgqa.set_decode_wait_limit_ns(5000)
    pgqa.set_decode_wait_limit_ns(0)   # back to the default; host only, no device touched
