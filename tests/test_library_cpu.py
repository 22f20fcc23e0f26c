"""Host-only checks of the C ABI: the library builds for sm_103a, loads without a GPU, exports
every symbol include/dg.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_grouped_fp8_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(lib, n), f"libdg.so does not export {n}"
    from moe_grouped_fp8_gb300 import _lib
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with include/*.h"


def test_binding_names_match_the_c_abi():
    from moe_grouped_fp8_gb300 import api
    for n in declared_functions():
        assert hasattr(api, n), n


def test_enum_values_match_header():
    src = open(os.path.join(ROOT, "include", "dg.h")).read()
    from moe_grouped_fp8_gb300 import _lib
    for name in ["DG_OK", "DG_ERR_INVALID_ARG", "DG_ERR_UNSUPPORTED", "DG_ERR_CUDA", "DG_SF_FP32", "DG_SF_UE8M0",
                 "DG_OUT_BF16", "DG_OUT_FP32", "DG_STATUS_BAD_INDEX", "DG_STATUS_COUNT_GT_CAP",
                 "DG_STATUS_K_NOT_ALIGNED", "DG_STATUS_K_OVERFLOW", "DG_STATUS_TIMEOUT", "DG_STATUS_TOO_MANY_RUNS",
                 "DG_MAX_GROUPS", "DG_MAX_M_BLOCKS", "DG_DEBUG_A_SCALE", "DG_DEBUG_B_SCALE", "DG_DEBUG_OUT",
                 "DG_DEBUG_CAST_IN", "DG_DEBUG_CAST_OUT"]:
        m = re.search(rf"\b{name}\s*=?\s*(\d+)", src)
        assert m, name
        assert int(m.group(1)) == getattr(_lib, name), name


def test_workspace_size(lib):
    assert lib.dg_workspace_size(2, 4, 0, 2048, 2048) == 4 * 2 * 128
    assert lib.dg_workspace_size(0, 32, 8192, 4096, 7168) == 0
    assert lib.dg_workspace_size(1, 32, 0, 6144, 7168) == 0


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: every case below fails validation first
FAKE_ODD = ctypes.c_void_p(0x10008)


@pytest.mark.parametrize("case", [
    ("quant_per_token K%128", lambda L: L.dg_quant_per_token_1x128(FAKE, 4, 100, 100, FAKE, FAKE, 0, 1e-30, None, 0, None)),
    ("quant_per_token ldx<K", lambda L: L.dg_quant_per_token_1x128(FAKE, 4, 256, 128, FAKE, FAKE, 0, 1e-30, None, 0, None)),
    ("quant_per_token fmt", lambda L: L.dg_quant_per_token_1x128(FAKE, 4, 256, 256, FAKE, FAKE, 7, 1e-30, None, 0, None)),
    ("quant_per_token null", lambda L: L.dg_quant_per_token_1x128(None, 4, 256, 256, FAKE, FAKE, 0, 1e-30, None, 0, None)),
    ("quant_per_token align", lambda L: L.dg_quant_per_token_1x128(FAKE_ODD, 4, 256, 256, FAKE, FAKE, 0, 1e-30, None, 0, None)),
    ("quant_per_token groups", lambda L: L.dg_quant_per_token_1x128(FAKE, 10, 256, 256, FAKE, FAKE, 0, 1e-30, FAKE, 3, None)),
    ("quant_block N%128", lambda L: L.dg_quant_block_128x128(FAKE, 2, 100, 256, FAKE, FAKE, 0, 1e-30, None)),
    ("quant_packed G", lambda L: L.dg_quant_per_token_1x128_packed(FAKE, 256, 256, FAKE, FAKE, 0, 1e-30, FAKE, 0, 8, None)),
    ("quant_packed counts", lambda L: L.dg_quant_per_token_1x128_packed(FAKE, 256, 256, FAKE, FAKE, 0, 1e-30, None, 2, 8, None)),
    ("quant_packed K", lambda L: L.dg_quant_per_token_1x128_packed(FAKE, 200, 256, FAKE, FAKE, 0, 1e-30, FAKE, 2, 8, None)),
    ("pack_rows bytes", lambda L: L.dg_pack_masked_rows(FAKE, 2, 8, 24, FAKE, FAKE, None)),
    ("pack_rows align", lambda L: L.dg_pack_masked_rows(FAKE_ODD, 2, 8, 32, FAKE, FAKE, None)),
    ("pack_rows G", lambda L: L.dg_pack_masked_rows(FAKE, 2000, 8, 32, FAKE, FAKE, None)),
    ("quant_channel C", lambda L: L.dg_quant_per_channel_128(FAKE, 256, 100, FAKE, 2, FAKE, FAKE, 1e-30, None, None)),
    ("quant_channel Kcap", lambda L: L.dg_quant_per_channel_128(FAKE, 200, 128, FAKE, 2, FAKE, FAKE, 1e-30, None, None)),
    ("quant_channel G", lambda L: L.dg_quant_per_channel_128(FAKE, 256, 128, FAKE, 0, FAKE, FAKE, 1e-30, None, None)),
    ("contig G", lambda L: L.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 128, 0, 256, 256, 0, None, 0, None, None)),
    ("contig G max", lambda L: L.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 128, 5000, 256, 256, 0, None, 0, None, None)),
    ("contig N", lambda L: L.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 128, 2, 200, 256, 0, None, 0, None, None)),
    ("contig out", lambda L: L.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 5, FAKE, 128, 2, 256, 256, 0, None, 0, None, None)),
    ("contig align", lambda L: L.dg_m_grouped_fp8_contiguous(FAKE_ODD, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 128, 2, 256, 256, 0, None, 0, None, None)),
    ("contig null idx", lambda L: L.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 0, None, 128, 2, 256, 256, 0, None, 0, None, None)),
    ("masked cap", lambda L: L.dg_m_grouped_fp8_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, -1, 256, 256, 0, 0, None, 0, None, None)),
    ("masked K", lambda L: L.dg_m_grouped_fp8_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 32, 256, 100, 0, 0, None, 0, None, None)),
    ("masked counts", lambda L: L.dg_m_grouped_fp8_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 0, None, 2, 32, 256, 256, 0, 0, None, 0, None, None)),
    ("kgrouped H", lambda L: L.dg_k_grouped_fp8_wgrad(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 2, 256, 256, 100, FAKE, 512, None, None)),
    ("kgrouped ws", lambda L: L.dg_k_grouped_fp8_wgrad(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 2, 256, 256, 256, FAKE, 100, None, None)),
    ("kgrouped ws null", lambda L: L.dg_k_grouped_fp8_wgrad(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 2, 256, 256, 256, None, 512, None, None)),
    ("kgrouped Kcap", lambda L: L.dg_k_grouped_fp8_wgrad(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 2, 200, 256, 256, FAKE, 512, None, None)),
    ("kgrouped sf align", lambda L: L.dg_k_grouped_fp8_wgrad(FAKE, FAKE_ODD, FAKE, FAKE, None, FAKE, FAKE, 2, 256, 256, 256, FAKE, 512, None, None)),
], ids=lambda c: c[0])
def test_invalid_arguments_rejected_on_host(lib, case):
    name, call = case
    rc = call(lib)
    assert rc == 1, (name, rc, lib.dg_last_error())
    assert lib.dg_last_error()


def test_too_large_is_unsupported(lib):
    rc = lib.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4096 * 128 + 1, 2, 256, 256, 0,
                                         None, 0, None, None)
    assert rc == 2, lib.dg_last_error()


def test_empty_problems_are_no_ops(lib):
    # zero rows / zero capacity enqueue nothing and succeed without a device
    assert lib.dg_quant_per_token_1x128(FAKE, 0, 256, 256, FAKE, FAKE, 0, 1e-30, None, 0, None) == 0
    assert lib.dg_m_grouped_fp8_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 0, 256, 256, 0, 0, None, 0, None,
                                       None) == 0
    assert lib.dg_m_grouped_fp8_contiguous(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 2, 256, 256, 0, None, 0, None,
                                           None) == 0
    assert lib.dg_quant_block_128x128(FAKE, 0, 256, 256, FAKE, FAKE, 0, 1e-30, None) == 0


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "moe_grouped_fp8_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".hpp", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt and "oracle.c" not in txt, f


def test_arg_log_records_every_call_before_its_checks(lib, tmp_path):
    """The argument log writes one line per call, with every argument by name, even for calls
    that fail validation (nothing here touches a device)."""
    path = tmp_path / "args.log"
    assert lib.dg_set_arg_log(str(path).encode()) == 0
    try:
        assert lib.dg_quant_per_token_1x128(FAKE, 4, 100, 100, FAKE, FAKE, 0, 1e-30, None, 0, None) == 1
        assert lib.dg_m_grouped_fp8_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 0, 256, 256, 192, 1, None, 0,
                                           None, None) == 0
        lib.dg_workspace_size(2, 4, 0, 2048, 2048)
    finally:
        assert lib.dg_set_arg_log(None) == 0
    lines = path.read_text().splitlines()
    assert len(lines) == 3, lines
    seq = [int(l.split()[0]) for l in lines]
    assert seq == sorted(seq) and len(set(seq)) == 3
    f0 = dict(kv.split("=", 1) for kv in lines[0].split()[2:])
    assert lines[0].split()[1] == "dg_quant_per_token_1x128"
    assert list(f0) == ["x", "M", "K", "ldx", "q", "sfa", "sf_format", "sf_zero", "row_counts", "G", "stream"]
    assert int(f0["x"], 16) == 0x10000 and f0["M"] == "4" and f0["K"] == "100" and f0["sf_format"] == "0"
    assert float(f0["sf_zero"]) == pytest.approx(1e-30, rel=1e-6)
    f1 = dict(kv.split("=", 1) for kv in lines[1].split()[2:])
    assert lines[1].split()[1] == "dg_m_grouped_fp8_masked"
    assert (f1["G"], f1["cap"], f1["N"], f1["K"], f1["expected_m"], f1["sf_format"]) == ("2", "0", "256", "256",
                                                                                         "192", "1")
    assert lines[2].split()[1] == "dg_workspace_size" and "N=2048" in lines[2]
    # stopped: later calls add nothing
    lib.dg_workspace_size(2, 4, 0, 2048, 2048)
    assert len(path.read_text().splitlines()) == 3


def test_arg_log_from_environment(tmp_path):
    """DG_ARG_LOG, read when the library loads, starts the log (fresh process)."""
    import subprocess
    import sys
    path = tmp_path / "env.log"
    code = ("from moe_grouped_fp8_gb300 import _lib; L = _lib.load(); "
            "L.dg_workspace_size(2, 3, 0, 256, 384); print(L.dg_debug_build())")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       env={**os.environ, "DG_ARG_LOG": str(path), "DG_DEBUG": "0"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "0"  # the release build
    assert path.read_text().split()[1:] == ["dg_workspace_size", "op=2", "G=3", "M=0", "N=256", "K=384"]
