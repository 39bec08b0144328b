"""The C-ABI library loads and exports every function include/nrm.h declares,
and rejects invalid arguments before touching a GPU (no GPU needed: the
pointers below are never dereferenced, and no call here reaches a launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nrm.h")

OK, NULL, SHAPE, DTYPE, ALIAS, VALUE, UNSUP, WS, DEVICE, LAUNCH, POINTER = range(11)


@pytest.fixture(scope="module")
def lib():
    import row_wise_normalization_reduce_gb300 as nrm
    if not os.path.exists(nrm.LIB_PATH):
        nrm.build()
    return nrm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_four_operators():
    names = declared_functions()
    for f in ("ln_fwd", "rms_fwd", "add_rms_fwd", "bn_fwd_train"):
        assert f in names


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"libnrm.so does not export {n}"


def test_status_strings(lib):
    for s in range(11):
        text = lib.nrm_status_string(s).decode()
        assert text and text != "unknown status"
    assert lib.nrm_status_string(999).decode() == "unknown status"


A = 0x10000  # fake, aligned addresses (never dereferenced)


def test_row_ops_validate_before_launch(lib):
    # null required pointers
    assert lib.ln_fwd(None, None, None, A, None, None, 4, 8, 1e-5, 0, None) == NULL
    assert lib.rms_fwd(A, None, None, None, 4, 8, 1e-5, 0, None) == NULL
    assert lib.add_rms_fwd(A, None, None, A * 4, A * 8, None, 4, 8, 1e-6, 2, None) == NULL
    # shapes, dtype, eps
    assert lib.ln_fwd(A, None, None, A * 4, None, None, -1, 8, 1e-5, 0, None) == SHAPE
    assert lib.ln_fwd(A, None, None, A * 4, None, None, 4, 0, 1e-5, 0, None) == SHAPE
    assert lib.ln_fwd(A, None, None, A * 4, None, None, 2 ** 40, 2 ** 40, 1e-5, 0, None) == SHAPE
    assert lib.ln_fwd(A, None, None, A * 4, None, None, 4, 8, 1e-5, 7, None) == DTYPE
    assert lib.ln_fwd(A, None, None, A * 4, None, None, 4, 8, -1.0, 0, None) == VALUE
    assert lib.ln_fwd(A, None, None, A * 4, None, None, 4, 8, float("nan"), 0, None) == VALUE
    assert lib.rms_fwd(A, None, A * 4, None, 4, 8, float("inf"), 1, None) == VALUE
    # misaligned to the element size
    assert lib.ln_fwd(A + 1, None, None, A * 4, None, None, 4, 8, 1e-5, 2, None) == VALUE
    assert lib.ln_fwd(A, None, None, A * 4, A * 8 + 2, None, 4, 8, 1e-5, 2, None) == VALUE
    # rows == 0 is a no-op that needs no device
    assert lib.ln_fwd(A, None, None, A * 4, None, None, 0, 8, 1e-5, 0, None) == OK
    assert lib.add_rms_fwd(A, A * 2, None, A * 3, A * 4, None, 0, 8, 1e-6, 2, None) == OK


def test_aliasing_rules(lib):
    rows, n = 4, 64
    tb = rows * n * 2
    x, res, ro, y = A, A + 4 * tb, A + 8 * tb, A + 12 * tb
    # y == x, or y overlapping x
    assert lib.ln_fwd(x, None, None, x, None, None, rows, n, 1e-5, 2, None) == ALIAS
    assert lib.ln_fwd(x, None, None, x + tb - 16, None, None, rows, n, 1e-5, 2, None) == ALIAS
    assert lib.rms_fwd(x, None, y, y + 16, rows, n, 1e-6, 2, None) == ALIAS
    # stats overlapping an input
    assert lib.ln_fwd(x, None, None, y, x + 64, None, rows, n, 1e-5, 2, None) == ALIAS
    # residual_out may be exactly residual, but not partially overlap it
    assert lib.add_rms_fwd(x, res, None, res + 16, y, None, rows, n, 1e-6, 2, None) == ALIAS
    assert lib.add_rms_fwd(x, res, None, ro, x, None, rows, n, 1e-6, 2, None) == ALIAS
    assert lib.add_rms_fwd(x, res, None, ro, ro, None, rows, n, 1e-6, 2, None) == ALIAS
    # valid calls get as far as the device query (no GPU in this container) or run
    st = lib.add_rms_fwd(x, res, None, res, y, None, rows, n, 1e-6, 2, None)
    assert st in (OK, DEVICE)


def bn_ws_formula(b, c, hw, es):
    # include/nrm.h: roundup16(8 * P) + 24 * C, P = batch * C * chunks per plane
    packs = -(-hw // (16 // es))
    chunks = b * c * -(-packs // 1024)
    return -(-8 * chunks // 16) * 16 + 24 * c


def test_bn_validation(lib):
    b, c, hw = 2, 3, 5
    need = lib.bn_fwd_train_workspace_size(b, c, hw, 0)
    assert need == bn_ws_formula(b, c, hw, 4) == 120
    for shape, dt, es in (((2, 3, 5000), 0, 4), ((3, 5, 9000), 2, 2), ((1, 1, 1), 1, 2)):
        assert lib.bn_fwd_train_workspace_size(*shape, dt) == bn_ws_formula(*shape, es)
    assert lib.bn_fwd_train_workspace_size(0, c, hw, 0) == 0
    assert lib.bn_fwd_train_workspace_size(b, c, hw, 9) == 0
    x, y, ws = A, A * 16, A * 64
    args = dict(g=None, be=None, sm=None, sr=None, rm=None, rv=None)

    def call(x=x, y=y, batch=b, C=c, HW=hw, eps=1e-5, mom=0.1, dt=0, ws=ws, wsb=need):
        return lib.bn_fwd_train(x, args["g"], args["be"], y, args["sm"], args["sr"], args["rm"],
                                args["rv"], batch, C, HW, eps, mom, dt, ws, wsb, None)

    assert call(x=None) == NULL
    assert call(batch=0) == SHAPE
    assert call(batch=1, HW=1) == SHAPE          # count 1: unbiased variance undefined
    assert call(eps=-1.0) == VALUE
    assert call(mom=1.5) == VALUE
    assert call(dt=5) == DTYPE
    assert call(dt=2) in (OK, DEVICE)            # bfloat16 data: valid
    assert call(ws=None) == WS
    assert call(wsb=need - 1) == WS
    assert call(ws=ws + 8) == WS
    assert call(y=x) == ALIAS
    assert call(ws=x) == ALIAS
    assert call() in (OK, DEVICE)


def test_bn_infer_validation(lib):
    b, c, hw = 2, 3, 5
    x, y, rm, rv = A, A * 16, A * 32, A * 33

    def call(x=x, y=y, rm=rm, rv=rv, batch=b, C=c, HW=hw, eps=1e-5, dt=0, g=None):
        return lib.bn_fwd_infer(x, g, None, y, rm, rv, batch, C, HW, eps, dt, None)

    assert call(batch=0, x=None, y=None) == OK    # empty batch: no pointer used
    assert call(x=None) == NULL
    assert call(rm=None) == NULL
    assert call(rv=None) == NULL
    assert call(batch=-1) == SHAPE
    assert call(C=0) == SHAPE
    assert call(eps=float("nan")) == VALUE
    assert call(dt=3) == DTYPE
    assert call(y=x) == ALIAS
    assert call(y=rm - 8) == ALIAS               # y overlaps the running mean
    assert call(x=x + 2, dt=0) == VALUE          # misaligned binary32 element
    assert call(dt=1) in (OK, DEVICE)
    assert call() in (OK, DEVICE)


def test_bn_bwd_validation(lib):
    b, c, hw = 2, 3, 5
    need = lib.bn_bwd_workspace_size(b, c, hw, 0)
    assert need == bn_ws_formula(b, c, hw, 4)
    assert lib.bn_bwd_workspace_size(b, 0, hw, 0) == 0
    dy, x, sm, sr, dx, ws = A, A * 16, A * 32, A * 33, A * 48, A * 64

    def call(dy=dy, x=x, sm=sm, sr=sr, dx=dx, dg=None, db=None, batch=b, C=c, HW=hw, dt=0,
             ws=ws, wsb=need):
        return lib.bn_bwd(dy, x, None, sm, sr, dx, dg, db, batch, C, HW, dt, ws, wsb, None)

    for kw in ({"dy": None}, {"x": None}, {"sm": None}, {"sr": None}, {"dx": None}):
        assert call(**kw) == NULL, kw
    assert call(batch=0) == SHAPE
    assert call(dt=7) == DTYPE
    assert call(ws=None) == WS
    assert call(wsb=need - 8) == WS
    assert call(dx=dy) == ALIAS
    assert call(dx=x + 8) == ALIAS
    assert call(dg=sm) == ALIAS                  # dgamma over the saved mean
    assert call(db=ws) == ALIAS                  # dbeta over the workspace
    assert call(dt=2) in (OK, DEVICE)
    assert call() in (OK, DEVICE)


def test_softmax_validation(lib):
    rows, n = 4, 64
    x, y, m, d = A, A * 4, A * 8, A * 9
    assert lib.softmax_fwd(None, y, None, None, rows, n, 0, None) == NULL
    assert lib.softmax_fwd(x, None, None, None, rows, n, 0, None) == NULL
    assert lib.softmax_fwd(None, None, None, None, 0, n, 0, None) == OK   # empty
    assert lib.softmax_fwd(x, y, None, None, rows, 0, 0, None) == SHAPE
    assert lib.softmax_fwd(x, y, None, None, rows, n, 4, None) == DTYPE
    assert lib.softmax_fwd(x, x + 64, None, None, rows, n, 2, None) == ALIAS
    assert lib.softmax_fwd(x, y, x, None, rows, n, 2, None) == ALIAS
    assert lib.softmax_fwd(x, y, m, m + 4, rows, n, 2, None) == ALIAS
    assert lib.softmax_fwd(x + 2, y, None, None, rows, n, 0, None) == VALUE
    assert lib.softmax_fwd(x, y, m, d, rows, n, 1, None) in (OK, DEVICE)


def test_force_plan_api(lib):
    assert lib.nrm_force_plan(99, 0, 0, 0, 0) == UNSUP
    assert lib.nrm_force_plan(-1, 0, 0, 0, 0) == UNSUP
    assert lib.nrm_force_plan(4, 256, 2, 17, 0) == UNSUP
    assert lib.nrm_force_plan(4, 256, 2, 2, 16) == UNSUP
    assert lib.nrm_force_plan(3, 256, 2, 0, 0) == OK
    assert lib.nrm_force_plan(4, 256, 2, 4, 2) == OK
    assert lib.nrm_force_plan(0, 0, 0, 0, 0) == OK
    old = lib.nrm_set_wait_limit(5)
    assert lib.nrm_set_wait_limit(old) == 5
    assert lib.nrm_set_pointer_checks(0) in (0, 1)


def test_product_path_has_no_oracle_dependency():
    # the package and the CUDA sources never name the oracle
    pkg = os.path.join(ROOT, "row_wise_normalization_reduce_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle." not in text, f


def _model_overlap(a, lda, wa, b, ldb, wb, rows):
    """Byte-level model of the library's overlap rule (exact for equal strides,
    outer bounds otherwise), for fake addresses."""
    ea, eb = a + (rows - 1) * lda + wa, b + (rows - 1) * ldb + wb
    if not (a < eb and b < ea):
        return False
    if lda != ldb or rows == 1:
        return True
    ra = set()
    for i in range(rows):
        ra.update(range(a + i * lda, a + i * lda + wa))
    return any(any(x in ra for x in range(b + j * ldb, b + j * ldb + wb)) for j in range(rows))


def test_sync_bn_validation(lib):
    b, c, hw = 2, 3, 5
    x, st, ws, y, parts, dy, dx = A, A * 16, A * 32, A * 48, A * 64, A * 80, A * 96
    assert lib.bn_fwd_partial_stats(None, st, b, c, hw, 0, ws, 256, None) == NULL
    assert lib.bn_fwd_partial_stats(x, st, b, c, hw, 0, ws, 8, None) == WS
    assert lib.bn_fwd_partial_stats(x, st + 4, b, c, hw, 0, ws, 256, None) == VALUE
    assert lib.bn_fwd_partial_stats(x, x + 8, b, c, hw, 0, ws, 256, None) == ALIAS
    assert lib.bn_fwd_partial_stats(x, st, b, c, hw, 0, ws, 256, None) in (OK, DEVICE)
    args = (None, None, None, None, None, None)
    assert lib.bn_fwd_apply_stats(x, None, None, y, parts, 0, *args[:4], b, c, hw, 1e-5, 0.1, 0,
                                  None) == SHAPE
    assert lib.bn_fwd_apply_stats(x, None, None, x, parts, 1, *args[:4], b, c, hw, 1e-5, 0.1, 0,
                                  None) == ALIAS
    assert lib.bn_fwd_apply_stats(x, None, None, y, parts, 2, *args[:4], b, c, hw, 1e-5, 2.0, 0,
                                  None) == VALUE
    assert lib.bn_fwd_apply_stats(x, None, None, y, parts, 2, *args[:4], b, c, hw, 1e-5, 0.1, 0,
                                  None) in (OK, DEVICE)
    assert lib.bn_bwd_partial_sums(dy, x, None, st, parts, b, c, hw, 0, ws, 256, None) == NULL
    assert lib.bn_bwd_partial_sums(dy, x, st, st + 64, parts, b, c, hw, 0, ws, 256,
                                   None) in (OK, DEVICE)
    assert lib.bn_bwd_apply_sums(dy, x, None, st, st + 64, parts, 2, b * hw - 1, dx, None, None,
                                 b, c, hw, 0, None) == SHAPE
    assert lib.bn_bwd_apply_sums(dy, x, None, st, st + 64, parts, 2, 2 * b * hw, dy, None, None,
                                 b, c, hw, 0, None) == ALIAS
    assert lib.bn_bwd_apply_sums(dy, x, None, st, st + 64, parts, 2, 2 * b * hw, dx, None, None,
                                 b, c, hw, 0, None) in (OK, DEVICE)


def test_host_pipe_validation(lib):
    rows, n = 8, 64
    x, r, ro, y = A, A * 2, A * 3, A * 4
    need = lib.add_rms_fwd_host_workspace_size(n, 2)
    assert need > 0 and lib.add_rms_fwd_host_workspace_size(0, 2) == 0
    ws = A * 1024
    call = lambda **k: lib.add_rms_fwd_host(k.get("x", x), k.get("r", r), None, k.get("ro", ro),
                                            k.get("y", y), None, k.get("rows", rows), n, 1e-6,
                                            k.get("dt", 2), k.get("ws", ws), k.get("wsb", need),
                                            None)
    assert call(rows=0, x=None) == OK
    assert call(x=None) == NULL
    assert call(dt=9) == DTYPE
    assert call(wsb=need - 1) == WS
    assert call(ws=ws + 16) == WS                 # not 256-byte aligned
    assert call(y=x) == ALIAS
    assert call(ro=r + 64) == ALIAS
    assert call(ro=r) in (OK, DEVICE)             # in place on the host
    assert call() in (OK, DEVICE)


def test_strided_alias_rule_matches_byte_model(lib):
    import random
    rng = random.Random(5)
    base = 1 << 20
    for _ in range(400):
        rows = rng.randint(1, 5)
        n = rng.randint(1, 12)
        ldx = n + rng.randint(0, 12)
        ldy = ldx if rng.random() < 0.7 else n + rng.randint(0, 12)
        off = rng.randint(-3 * ldx, 3 * ldx)
        x = base
        y = base + 4 * off
        if y <= 0:
            continue
        want = _model_overlap(x, 4 * ldx, 4 * n, y, 4 * ldy, 4 * n, rows)
        st = lib.rms_fwd_ld(x, ldx, None, y, ldy, None, rows, n, 1e-6, 0, None)
        assert (st == ALIAS) == want, (rows, n, ldx, ldy, off, st)


def test_strided_validation(lib):
    x, y = A, A * 64
    assert lib.ln_fwd_ld(x, 7, None, None, y, 8, None, None, 3, 8, 1e-5, 0, None) == SHAPE
    assert lib.ln_fwd_ld(x, 8, None, None, y, 7, None, None, 3, 8, 1e-5, 0, None) == SHAPE
    assert lib.softmax_fwd_ld(x, 2 ** 62, y, 8, None, None, 3, 8, 0, None) == SHAPE
    # y in the columns next to x in one padded buffer: allowed
    assert lib.ln_fwd_ld(x, 16, None, None, x + 32, 16, None, None, 3, 8, 1e-5, 0, None) in (OK, DEVICE)
    # ... but not one column further left
    assert lib.ln_fwd_ld(x, 16, None, None, x + 28, 16, None, None, 3, 8, 1e-5, 0, None) == ALIAS
    # in-place residual needs the same stride
    assert lib.add_rms_fwd_ld(x, 8, y, 16, None, y, 12, y + 4096, 8, None, 3, 8, 1e-6, 0,
                              None) == ALIAS
    assert lib.add_rms_fwd_ld(x, 8, y, 16, None, y, 16, y + 4096, 8, None, 3, 8, 1e-6, 0,
                              None) in (OK, DEVICE)


def test_header_compiles_as_c(tmp_path):
    # include/nrm.h is a C interface: it must compile as strict C11 (and C++)
    # with every warning an error
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = next((p for p in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda")
                     if p and os.path.exists(os.path.join(p, "include", "cuda_runtime_api.h"))), None)
    if not gcc or not cuda_inc:
        pytest.skip("gcc or the CUDA headers not found")
    src = tmp_path / "use_nrm.c"
    src.write_text('#include "nrm.h"\n'
                   "int main(void) { return bn_fwd_train_workspace_size(1, 1, 2, NRM_F32) == 0; }\n")
    inc = ["-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda_inc, "include")]
    for lang in (["-x", "c", "-std=c11", "-pedantic"], ["-x", "c++", "-std=c++17"]):
        r = subprocess.run([gcc, *lang, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", *inc, str(src)],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
