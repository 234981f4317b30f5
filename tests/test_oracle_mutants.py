"""The oracle's pins have teeth: plausible mistakes planted in the oracle each fail at least one of them.

Each mutant is the oracle with one edit of the kind a careless restatement of the pages' formulas would make
(a dropped term, a wrong index or base, an off-by-one, a wrong search or tie rule).  C mutants are compiled on
the CPU and the oracle package is pointed at the result; Python mutants are a mutated copy of the package's
source whose edited function replaces the oracle's.  The pins then run until one fails.  The unmutated
source, through the same runner, must pass every pin -- so a mutant that survives means a pin is missing,
not that the runner is broken.  Nothing here touches a GPU.
"""
import inspect
import itertools
import os
import shutil
import types

import pytest

import oracle
import test_cascade_host
import test_extra_pins
import test_oracle_pins as pins
import test_selection_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

# (what the mistake is, the exact source text it replaces, the replacement)
MUTANTS = [
    ("page resolution drops first_page_offset",
     "int64_t t = (int64_t)first_page_offset[r] + i;", "int64_t t = i;"),
    ("page resolution drops the entry within the page",
     "return (int64_t)indices[slot] * page_size + entry;", "return (int64_t)indices[slot] * page_size;"),
    ("page resolution ignores the page table (identity pages)",
     "return (int64_t)indices[slot] * page_size + entry;", "return slot * page_size + entry;"),
    ("scores lose the softmax scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("scores use V instead of K",
     "dot += q[d] * ora_elem(p->k_pool, p->dtype, base + d);", "dot += q[d] * ora_elem(p->v_pool, p->dtype, base + d);"),
    ("query head h reads KV head h % Hkv instead of h / G",
     "ora_attend_range(&p, qd, scale, r, h / group, 0, L,", "ora_attend_range(&p, qd, scale, r, h % num_kv_heads, 0, L,"),
    ("attention LSE in natural log instead of base 2",
     "*lse2 = (m + log(den)) / M_LN2;", "*lse2 = m + log(den);"),
    ("merge weights use exp instead of exp2",
     "double w = (l == -INFINITY) ? 0.0 : exp2(l - m);", "double w = (l == -INFINITY) ? 0.0 : exp(l - m);"),
    ("merge LSE in natural log", "lse_out[(int64_t)r * num_heads + h] = log2(wsum) + m;",
     "lse_out[(int64_t)r * num_heads + h] = log(wsum) + m;"),
    ("chunk end one token short",
     "int64_t i1 = (k + 1) * pages_per_chunk * page_size - first_page_offset[r];",
     "int64_t i1 = (k + 1) * pages_per_chunk * page_size - first_page_offset[r] - 1;"),
    ("chunk start ignores first_page_offset",
     "int64_t i0 = k * pages_per_chunk * page_size - first_page_offset[r];",
     "int64_t i0 = k * pages_per_chunk * page_size;"),
    ("plan takes the smallest size reaching the target, not the largest",
     "if (ora_num_chunks(indptr, batch, p) * num_kv_heads * q_groups >= target_ctas)\n                ppc = p;",
     "if (ora_num_chunks(indptr, batch, p) * num_kv_heads * q_groups >= target_ctas) {\n"
     "                ppc = p;\n                break;\n            }"),
    ("plan compares > instead of >= against the target",
     "* num_kv_heads * q_groups >= target_ctas)", "* num_kv_heads * q_groups > target_ctas)"),
    ("plan drops the one-chunk floor for empty requests", "n += c > 1 ? c : 1;", "n += c;"),
    ("seq_len ignores last_page_len",
     "return (pages - 1) * page_size + last_page_len[r] - first_page_offset[r];",
     "return pages * page_size - first_page_offset[r];"),
    ("validation rejects an exactly full last page",
     "if (last_page_len[r] < 1 || last_page_len[r] > page_size)",
     "if (last_page_len[r] < 1 || last_page_len[r] >= page_size)"),
    ("validation accepts page ids past the pool",
     "if (indices[j] < 0 || (int64_t)indices[j] >= num_pages)", "if (indices[j] < 0 || (int64_t)indices[j] > num_pages)"),
    ("binary16 exponent bias off by one",
     "mag = ldexp((double)(1024 + frac), expo - 25);", "mag = ldexp((double)(1024 + frac), expo - 24);"),
    ("binary16 subnormal scale off by one", "mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    ("bfloat16 placed in the wrong half of the binary32", "uint32_t bits = (uint32_t)b << 16;",
     "uint32_t bits = (uint32_t)b << 15;"),
]


OracleSrc = os.path.join(os.path.dirname(oracle.__file__), "__init__.py")
# pins only: tests that compare the oracle with the library's own host code are parity checks, not pins
SELECTION = (test_selection_pins,)
DETECTION = ((test_cascade_host, {"test_detect_rules_by_hand", "test_detect_tie_goes_to_the_group_met_first"}),
             pins)

# (what the mistake is, the oracle functions it changes, the exact source text, the replacement, the pin
# modules to run)
PY_MUTANTS = [
    ("detection: on a tie the later group wins", ("cascade_detect_ref",),
     "        if score > best_score:", "        if score >= best_score:", DETECTION),
    ("detection: the shared span may cover a member's last page", ("cascade_detect_ref",),
     "cap = min(ip[r + 1] - ip[r] - 1 for r in mem)", "cap = min(ip[r + 1] - ip[r] for r in mem)", DETECTION),
    ("detection: windows that start mid-page join a group", ("cascade_detect_ref",),
     "if fp[r] != 0 or pages < 2:", "if pages < 2:", DETECTION),
    ("selection: rows one past each block", ("selection_rows_ref",),
     "out.append(base + j * block_size + e)", "out.append(base + j * block_size + e + 1)", SELECTION),
    ("selection: request stride ignored", ("selection_rows_ref",),
     "        base = r * request_stride\n", "        base = 0\n", SELECTION),
    ("selection: final block left out", ("selection_rows_ref",),
     "        for e in range(last):\n            out.append(base + (nb - 1) * block_size + e)\n", "", SELECTION),
    ("block-granular table puts the final block first", ("selection_pages_ref",),
     "pages += [r * blocks_per_request + j for j in sel] + [r * blocks_per_request + nb - 1]",
     "pages += [r * blocks_per_request + nb - 1] + [r * blocks_per_request + j for j in sel]", SELECTION),
    ("second K stream: the extra score term dropped", ("attention_extra", "partials_extra"),
     "s = scale * (qr @ K.T + qer @ Ke.T)", "s = scale * (qr @ K.T)", (test_extra_pins,)),
    ("second K stream: LSE in natural log", ("attention_extra", "partials_extra"),
     "return (w / tot) @ V, (m[:, 0] + np.log(tot[:, 0])) / np.log(2.0)",
     "return (w / tot) @ V, m[:, 0] + np.log(tot[:, 0])", (test_extra_pins,)),
]


def _pin_calls(modules=(pins,)):
    """Every pin of `modules` (a module, or (module, the names of the pins to take)) as (name, function,
    kwargs), parametrize marks expanded; pins that take fixtures are left out."""
    calls = []
    for mod in modules:
        mod, only = mod if isinstance(mod, tuple) else (mod, None)
        calls += [c for c in _module_pin_calls(mod) if only is None or c[0] in only]
    return calls


def _module_pin_calls(mod):
    calls = []
    for name, fn in inspect.getmembers(mod, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != mod.__name__:
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = [n.strip() for n in mark.args[0].split(",")] if isinstance(mark.args[0], str) else mark.args[0]
            values = [v if len(names) > 1 else (v,) for v in mark.args[1]]
            grids.append([dict(zip(names, v)) for v in values])
        params = set(inspect.signature(fn).parameters)
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            if set(kw) == params:
                calls.append((name, fn, kw))
    return calls


def _first_failing_pin(src_text, workdir, tag):
    """Compile `src_text` as the oracle, point the oracle package at it, and return the name of the first pin
    that fails (None if all pass)."""
    src = os.path.join(workdir, f"{tag}.c")
    with open(src, "w") as f:
        f.write(src_text)
    saved = (oracle._SRC, oracle._LIB_PATH, oracle._lib)
    oracle._SRC, oracle._LIB_PATH, oracle._lib = src, os.path.join(workdir, f"lib{tag}.so"), None
    try:
        oracle.build(force=True)  # outside the pins: a mutant that does not compile is an error, not a catch
        oracle.lib()
        return _run_pins(_pin_calls())
    finally:
        oracle._SRC, oracle._LIB_PATH, oracle._lib = saved


def _run_pins(calls):
    for name, fn, kw in calls:
        try:
            fn(**kw)
        except Exception:  # noqa: BLE001 -- any failure (assertion or error) counts as caught
            return f"{name}{kw or ''}"
    return None


def _python_mutant_catch(text, names, modules, workdir, tag):
    """Load `text` as a copy of the oracle package (beside a copy of its C source), swap its functions
    `names` into the oracle, and return the first pin of `modules` that fails (None if all pass)."""
    d = os.path.join(workdir, tag)
    os.makedirs(d, exist_ok=True)
    shutil.copy(SRC, os.path.join(d, "pa_oracle.c"))
    path = os.path.join(d, "__init__.py")
    with open(path, "w") as f:
        f.write(text)
    mod = types.ModuleType("oracle_" + tag)
    mod.__file__ = path
    exec(compile(text, path, "exec"), mod.__dict__)
    saved = {n: getattr(oracle, n) for n in names}
    try:
        for n in names:
            setattr(oracle, n, getattr(mod, n))
        return _run_pins(_pin_calls(modules))
    finally:
        for n, f in saved.items():
            setattr(oracle, n, f)


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is needed to compile the oracle")
    return str(tmp_path_factory.mktemp("oracle_mutants"))


def test_unmutated_oracle_passes_every_pin_through_the_runner(workdir):
    text = open(SRC).read()
    assert len(_pin_calls()) >= 40
    assert _first_failing_pin(text, workdir, "clean") is None


@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_oracle_mistake_fails_a_pin(workdir, what, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation target not found exactly once: {old!r}"
    tag = "m%08x" % (abs(hash(what)) & 0xFFFFFFFF)
    caught = _first_failing_pin(text.replace(old, new), workdir, tag)
    assert caught is not None, f"no pin catches: {what}"
    print(f"{what}: caught by {caught}")


def test_unmutated_python_oracle_passes_every_pin_through_the_runner(workdir):
    text = open(OracleSrc).read()
    names = sorted({n for m in PY_MUTANTS for n in m[1]})
    modules = tuple({id(m): m for mut in PY_MUTANTS for m in mut[4]}.values())
    assert len(_pin_calls(modules)) >= 50
    assert _python_mutant_catch(text, names, modules, workdir, "pyclean") is None


@pytest.mark.parametrize("what,names,old,new,modules", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_python_oracle_mistake_fails_a_pin(workdir, what, names, old, new, modules):
    text = open(OracleSrc).read()
    assert text.count(old) == 1, f"mutation target not found exactly once: {old!r}"
    tag = "p%08x" % (abs(hash(what)) & 0xFFFFFFFF)
    caught = _python_mutant_catch(text.replace(old, new), names, modules, workdir, tag)
    assert caught is not None, f"no pin catches: {what}"
    print(f"{what}: caught by {caught}")
