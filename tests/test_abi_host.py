"""The C ABI on the host, without a GPU: exports, chunk planning, validation.

No call here launches GPU work; the only entry points called are the
host-only ones (kvx_validate, kvx_plan_chunks, kvx_default_launch, the
validation level, status strings) and error paths that return before any
CUDA call.
"""

import ctypes
import glob
import os
import re
import subprocess
import sys
import types

import numpy as np
import pytest

import oracle
import workloads as W
from expert_host_block_gb300 import build as kbuild
from expert_host_block_gb300 import kvx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session", autouse=True)
def _built():
    kbuild.build()


def _declared():
    names = set()
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(kvx_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_what_binding_lists():
    assert _declared() == sorted(kvx.EXPORTS)


# The boundary calls (the batch copy, the reusable descriptor buffers, the
# completion read, the direct baseline) and the comment block written right
# above each declaration.
BOUNDARY_CALLS = ("kvx_copy_batch", "kvx_copy_batch_ex", "kvx_desc_buf_create", "kvx_upload_descriptors",
                  "kvx_copy_uploaded", "kvx_copy_uploaded_ex", "kvx_desc_buf_info", "kvx_desc_buf_destroy",
                  "kvx_stream_check", "kvx_status_string", "kvx_copy_batch_memcpy", "kvx_copy_contiguous")
PAGE = re.compile(r"(PegaFlow issue #408|vLLM PR #42212 report|FreeToken issue #751)[^§]{0,80}§")


def _comment_above(text, name):
    m = re.search(r"\b" + name + r"\s*\(", re.sub(r"/\*.*?\*/", lambda c: " " * len(c.group()), text, flags=re.S))
    assert m, name
    end = text.rfind("*/", 0, m.start())
    start = text.rfind("/*", 0, end)
    between = text[end + 2:m.start()]
    assert "/*" not in between and ";" not in between, f"{name}: no comment block right above it"
    return text[start:end + 2]


def test_boundary_declarations_cite_a_page_and_section():
    text = open(os.path.join(ROOT, "include", "kvx.h")).read()
    for name in BOUNDARY_CALLS:
        block = " ".join(re.sub(r"^\s*\*(?!/)", " ", _comment_above(text, name), flags=re.M).split())
        assert PAGE.search(block), f"{name}: its comment names no page and section"
    # the one entry point with no counterpart on the pages says so instead
    noalloc = text[text.index("a batch copy that allocates nothing"):text.index("kvx_copy_batch_noalloc(")]
    noalloc = " ".join(re.sub(r"^\s*\*(?!/)", " ", noalloc, flags=re.M).split())
    assert "The pages have no counterpart" in noalloc


def test_library_exports_every_declared_symbol():
    lib = kvx.lib()
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", kvx.LIB_PATH], capture_output=True, text=True).stdout
    defined = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(_declared()) <= defined


def test_version_and_status_strings():
    assert kvx.kvx_version() == kvx.KVX_VERSION == 4
    names = [kvx.status_string(s) for s in range(10)]
    assert names[0] == "KVX_OK" and names[7] == "KVX_ERR_TIMEOUT" and names[9] == "KVX_ERR_CAPTURE"
    assert kvx.status_string(99) == "KVX_ERR_UNKNOWN"


# ---- chunk planning --------------------------------------------------------

def _apply(pool_dst, pool_src, so, do, sz):
    oracle.copy_batch(pool_dst, pool_src, so, do, sz)


@pytest.mark.parametrize("seed", range(4))
def test_chunk_table_moves_the_same_bytes(seed):
    """Applying the chunk records gives the oracle's result for the descriptors."""
    g = np.random.default_rng(seed)
    pool = 24 << 20
    src = g.integers(0, 256, pool, dtype=np.uint8)
    dst0 = g.integers(0, 256, pool, dtype=np.uint8)
    n = 200
    slot = 96 * 1024
    sizes = (8 * g.integers(0, 80 * 1024 // 8, n)).astype(np.uint64)
    sizes[:5] = [0, 8, 16384, 16392, 16384 * 3]
    so = (g.permutation(pool // slot)[:n] * slot + 8 * g.integers(0, 2, n)).astype(np.uint64)
    do = (g.permutation(pool // slot)[:n] * slot + 8 * g.integers(0, 2, n)).astype(np.uint64)
    base_s, base_d = 1 << 40, 1 << 41
    t = kvx.kvx_plan_chunks(so + base_s, do + base_d, sizes)
    assert t.size == int(sum(-(-int(z) // 16384) for z in sizes))
    assert np.all(t["len"] <= kvx.KVX_CHUNK_BYTES) and np.all(t["len"] > 0)
    # each chunk stays inside its descriptor, and chunk offsets line up
    i = t["desc"].astype(np.int64)
    assert np.all(t["src"] - (so[i] + base_s) == t["dst"] - (do[i] + base_d))
    assert np.all(t["src"] - (so[i] + base_s) + t["len"] <= sizes[i])
    assert np.all(t["reserved"] == 0)
    want = dst0.copy()
    _apply(want, src, so, do, sizes)
    got = dst0.copy()
    _apply(got, src, t["src"] - base_s, t["dst"] - base_d, t["len"].astype(np.uint64))
    assert np.array_equal(got, want)


def test_parallel_pack_matches_single_thread(tmp_path):
    """A table of >= 32,768 records is packed by the worker pool in descriptor ranges; it must equal the
    single-threaded table record for record."""
    code = ("import numpy as np\n"
            "from expert_host_block_gb300 import kvx\n"
            "g = np.random.default_rng(5)\n"
            "n = 16000\n"
            "z = (8 * g.integers(0, 80 * 1024 // 8, n)).astype(np.uint64)\n"
            "s = np.uint64(1 << 40) + np.arange(n, dtype=np.uint64) * np.uint64(1 << 20) + np.uint64(8) * g.integers(0, 2, n).astype(np.uint64)\n"
            "d = np.uint64(1 << 41) + np.arange(n, dtype=np.uint64) * np.uint64(1 << 20)\n"
            "t = kvx.kvx_plan_chunks(s, d, z)\n"
            f"np.save(r'{tmp_path}/' + __import__('os').environ['KVX_PACK_THREADS'] + '.npy', t.view(np.uint8))\n"
            "print(t.size)\n")
    a = _run_with_env(code, KVX_PACK_THREADS="0")
    b = _run_with_env(code, KVX_PACK_THREADS="3")
    assert a.returncode == 0 and b.returncode == 0, a.stderr + b.stderr
    assert int(a.stdout) >= 32768 and a.stdout == b.stdout
    assert np.array_equal(np.load(tmp_path / "0.npy"), np.load(tmp_path / "3.npy"))


def test_moe_chunk_count_closed_form(golden):
    """1 MiB / 16 KiB + 128 KiB / 16 KiB + 1 + 512 KiB / 16 KiB + ceil(68 KiB / 16 KiB) + 1 = 111."""
    rows = [int(x) for x in golden("moe_banks.txt")["row_bytes"]]
    m = W.MoeGather()
    b = m.next_call()
    t = kvx.kvx_plan_chunks(b.src_off + (1 << 40), b.dst_off + (1 << 41), b.sizes)
    assert 64 + 8 + 1 + 32 + 5 + 1 == 111
    assert t.size == 32 * 111 == 3552
    assert int(t["len"].astype(np.int64).sum()) == 32 * sum(rows)


def test_plan_empty_and_zero_sizes():
    assert kvx.kvx_plan_chunks([], [], []).size == 0
    t = kvx.kvx_plan_chunks([0, 8], [0, 16], [0, 0])
    assert t.size == 0


# ---- validation ------------------------------------------------------------

def _ok_batch():
    return (np.array([1 << 20, 2 << 20], np.uint64), np.array([3 << 20, 4 << 20], np.uint64),
            np.array([4096, 8], np.uint64))


def test_validate_accepts_good_batch():
    s, d, z = _ok_batch()
    for level in (0, 1):
        assert kvx.kvx_validate(s, d, z, None, kvx.KVX_H2D, level) == kvx.KVX_OK


@pytest.mark.parametrize("field,value,status", [
    ("size", 4100, kvx.KVX_ERR_ALIGN),
    ("size", 12, kvx.KVX_ERR_ALIGN),
    ("src", (1 << 20) + 4, kvx.KVX_ERR_ALIGN),
    ("dst", (3 << 20) + 1, kvx.KVX_ERR_ALIGN),
    ("src", 0, kvx.KVX_ERR_INVALID_ARG),
    ("dst", 0, kvx.KVX_ERR_INVALID_ARG),
    ("src", (1 << 64) - 8, kvx.KVX_ERR_INVALID_ARG),
])
def test_validate_rejects(field, value, status):
    s, d, z = _ok_batch()
    {"size": z, "src": s, "dst": d}[field][0] = value
    assert kvx.kvx_validate(s, d, z, None, kvx.KVX_D2D, 0) == status
    assert kvx.last_error()


def test_validate_zero_size_ignores_addresses():
    assert kvx.kvx_validate([0, 3], [0, 5], [0, 0], None, kvx.KVX_H2D, 1) == kvx.KVX_OK


def test_validate_bad_dir_and_level():
    s, d, z = _ok_batch()
    assert kvx.kvx_validate(s, d, z, None, 3, 0) == kvx.KVX_ERR_INVALID_ARG
    assert kvx.kvx_validate(s, d, z, None, -1, 0) == kvx.KVX_ERR_INVALID_ARG
    assert kvx.kvx_validate(s, d, z, None, kvx.KVX_H2D, 3) == kvx.KVX_ERR_INVALID_ARG


def test_validate_null_arrays():
    L = kvx.lib()
    assert L.kvx_validate(None, None, None, 4, 0, 0) == kvx.KVX_ERR_INVALID_ARG
    assert L.kvx_validate(None, None, None, 0, 0, 0) == kvx.KVX_OK


def test_validate_overlap_only_at_level_1():
    s = np.array([1 << 20, 2 << 20], np.uint64)
    d = np.array([3 << 20, (3 << 20) + 4088], np.uint64)  # second starts 8 bytes before the first ends
    z = np.array([4096, 4096], np.uint64)
    assert kvx.kvx_validate(s, d, z, None, kvx.KVX_D2D, 0) == kvx.KVX_OK
    assert kvx.kvx_validate(s, d, z, None, kvx.KVX_D2D, 1) == kvx.KVX_ERR_OVERLAP
    d2 = np.array([3 << 20, (3 << 20) + 4096], np.uint64)  # touching, not overlapping
    assert kvx.kvx_validate(s, d2, z, None, kvx.KVX_D2D, 1) == kvx.KVX_OK
    # a destination overlapping a source of the batch
    s3 = np.array([(3 << 20) + 8, 2 << 20], np.uint64)  # inside the second destination
    assert kvx.kvx_validate(s3, d2 - np.uint64(4096), z, None, kvx.KVX_D2D, 1) == kvx.KVX_ERR_OVERLAP


def test_validate_overlap_matches_oracle_disjointness():
    g = np.random.default_rng(3)
    for _ in range(300):
        n = int(g.integers(1, 7))
        d = (8 * g.integers(1, 40, n)).astype(np.uint64) + np.uint64(1 << 30)
        z = (8 * g.integers(0, 6, n)).astype(np.uint64)
        s = (8 * g.integers(1, 40, n)).astype(np.uint64) + np.uint64(1 << 20)  # far from d
        want = kvx.KVX_OK if oracle.ranges_disjoint(d, z) else kvx.KVX_ERR_OVERLAP
        assert kvx.kvx_validate(s, d, z, None, kvx.KVX_D2D, 1) == want


def test_capacity_limit():
    # one descriptor of (KVX_MAX_CHUNKS + 1) * 16 KiB
    z = np.array([(kvx.KVX_MAX_CHUNKS + 1) * kvx.KVX_CHUNK_BYTES], np.uint64)
    assert kvx.kvx_validate([1 << 20], [1 << 40], z, None, kvx.KVX_D2D, 0) == kvx.KVX_ERR_CAPACITY
    z = np.array([kvx.KVX_MAX_CHUNKS * kvx.KVX_CHUNK_BYTES], np.uint64)
    assert kvx.kvx_validate([1 << 20], [1 << 40], z, None, kvx.KVX_D2D, 0) == kvx.KVX_OK


def test_huge_size_without_address_wrap_is_a_capacity_error():
    # a size within 16 KiB of 2^64 whose address does not wrap
    z = np.array([(1 << 64) - 16384 + 8], np.uint64)
    assert kvx.kvx_validate([8], [16], z, None, kvx.KVX_D2D, 0) == kvx.KVX_ERR_CAPACITY
    z = np.array([4096, 1 << 41], np.uint64)
    assert kvx.kvx_validate([1 << 20, 1 << 21], [1 << 30, 1 << 31], z, None, kvx.KVX_D2D, 0) == \
        kvx.KVX_ERR_CAPACITY
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_plan_chunks([8], [16], [(1 << 64) - 16384 + 8])
    assert e.value.status == kvx.KVX_ERR_CAPACITY


def test_copy_batch_rejects_before_any_cuda_call():
    s, d, z = _ok_batch()
    z[1] = 12
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_copy_batch(s, d, z, None, kvx.KVX_H2D, 0, None)
    assert e.value.status == kvx.KVX_ERR_ALIGN
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_copy_batch(s, d, z, None, kvx.KVX_H2D, -1, None)
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_copy_batch_memcpy(s, d, z, None, 7, None)
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    # n == 0 is a no-op that needs no device
    kvx.kvx_copy_batch([], [], [], None, kvx.KVX_H2D, 0, None)


@pytest.mark.parametrize("launch", [
    {"variant": 4}, {"variant": "stage", "stages": 6}, {"threads": 1024}, {"threads": 96}, {"unroll": 3},
    {"stages": 13},
    {"store_policy": 3}, {"cta_budget": -2}, {"assign": 3}, {"assign": -1},
])
def test_copy_batch_ex_rejects_bad_launch(launch):
    s, d, z = _ok_batch()
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_copy_batch_ex(s, d, z, None, kvx.KVX_D2D, launch, None)
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG


def test_default_launch_table():
    for dname in ("h2d", "d2h", "d2d"):
        for mean in (8, 4096, 16384):
            l = kvx.kvx_default_launch(dname, mean)
            assert l["variant"] in (kvx.KVX_VARIANT_LDG, kvx.KVX_VARIANT_BULK)
            assert l["cta_budget"] > 0 and l["threads"] in (128, 256, 512)
            assert l["unroll"] in (2, 4, 8) and 2 <= l["stages"] <= 12
            # units from a counter over the host link, by position for D2D
            want = kvx.KVX_ASSIGN_STATIC if dname == "d2d" else kvx.KVX_ASSIGN_DYNAMIC
            assert l["assign"] == want
    with pytest.raises(kvx.KvxError):
        kvx.kvx_default_launch(5, 4096)


def test_validate_level_setting():
    kvx.kvx_set_validate_level(1)
    assert kvx.kvx_get_validate_level() == 1
    kvx.kvx_set_validate_level(0)
    with pytest.raises(kvx.KvxError):
        kvx.kvx_set_validate_level(3)


@pytest.mark.parametrize("var,val", [("KVX_VARIANT", "tma"), ("KVX_VALIDATE", "yes"),
                                     ("KVX_CTA_BUDGET", "-4"), ("KVX_CTA_BUDGET", "12x"),
                                     ("KVX_PACK_THREADS", "many"), ("KVX_PACK_THREADS", "99"),
                                     ("KVX_NVTX", "on"), ("KVX_NVTX", "2"), ("KVX_PDL", "yes"),
                                     ("KVX_PDL", "2")])
def test_unknown_env_values_are_errors(var, val):
    code = ("from expert_host_block_gb300 import kvx\n"
            "try:\n"
            "    kvx.kvx_copy_batch([8], [16], [8], None, 0, 0, None)\n"
            "except kvx.KvxError as e:\n"
            "    print(e.status, e)\n")
    env = dict(os.environ, **{var: val})
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    assert out.stdout.startswith(f"{kvx.KVX_ERR_INVALID_ARG} "), out.stdout + out.stderr
    assert var in out.stdout


def test_descriptors_helper_fill_and_capacity():
    d = kvx.Descriptors(4).set([8, 16], [24, 32], [8, 8])
    assert d.n == 2 and list(d.src[:2]) == [8, 16] and list(d.sizes[:2]) == [8, 8]
    with pytest.raises(ValueError):
        d.set([8] * 5, [16] * 5, [8] * 5)
    d.sizes[1] = 12  # refilled in place: validation still applies
    with pytest.raises(kvx.KvxError) as e:
        d.copy_batch("h2d")
    assert e.value.status == kvx.KVX_ERR_ALIGN


def test_transfer_host_paths():
    t = kvx.Transfer()
    assert t.poll() is True and t.progress() == (0, 0)  # nothing started: done
    with pytest.raises(kvx.KvxError) as e:
        t.start([1 << 20], [1 << 30], [12], "h2d", 4)
    assert e.value.status == kvx.KVX_ERR_ALIGN
    t.start([], [], [], "h2d", 4)  # an empty transfer needs no device
    assert t.poll() is True
    t.close()


def test_auto_path_rules():
    M = 1 << 20
    # a few large ranges: DMA
    assert kvx.kvx_auto_path([1 << 30], [1 << 40], [4 * M], None, "h2d") == "dma"
    assert kvx.kvx_auto_path([1 << 30], [1 << 40], [256 << 10], None, "h2d") == "dma"
    assert kvx.kvx_auto_path([1 << 30] * 1, [1 << 40], [M], None, "h2d", "tail") == "dma"
    # 16 ranges of 1 MiB: the kernel for throughput, DMA (no SMs) for the tail
    s = (1 << 30) + 2 * M * np.arange(16, dtype=np.uint64)
    d = (1 << 40) + 2 * M * np.arange(16, dtype=np.uint64)
    assert kvx.kvx_auto_path(s, d, np.full(16, M), None, "h2d") == "kernel_ldg"
    assert kvx.kvx_auto_path(s, d, np.full(16, M), None, "h2d", "tail") == "dma"
    # 4 ranges of 1 MiB: DMA for both
    assert kvx.kvx_auto_path(s[:4], d[:4], np.full(4, M), None, "h2d") == "dma"
    # adjacent descriptors merge into one large range: DMA
    s = (1 << 30) + 4096 * np.arange(1024, dtype=np.uint64)
    d = (1 << 40) + 4096 * np.arange(1024, dtype=np.uint64)
    assert kvx.kvx_auto_path(s, d, np.full(1024, 4096), None, "d2d") == "dma"
    # shuffled small descriptors: the kernel, by policy
    g = np.random.default_rng(1)
    s = (1 << 30) + 4096 * g.permutation(4096)[:1024].astype(np.uint64)
    assert kvx.kvx_auto_path(s, d, np.full(1024, 4096), None, "h2d") == "kernel_ldg"
    assert kvx.kvx_auto_path(s, d, np.full(1024, 4096), None, "h2d", "tail") == "kernel_bulk"
    # 17 large ranges: too many to submit one by one, for either policy
    s = (1 << 30) + 2 * M * np.arange(17, dtype=np.uint64)
    d = (1 << 40) + 2 * M * np.arange(17, dtype=np.uint64)
    assert kvx.kvx_auto_path(s, d, np.full(17, M), None, "h2d") == "kernel_ldg"
    assert kvx.kvx_auto_path(s, d, np.full(17, M), None, "h2d", "tail") == "kernel_bulk"
    # two ranges with a mean below 2 x 256 KiB: kernel
    assert kvx.kvx_auto_path([1 << 30, 1 << 31], [1 << 40, 1 << 41], [256 << 10, 8], None, "h2d") == "kernel_ldg"
    # throughput takes the calibrated table's kernel: LDG for 256 MiB of aligned 16 KiB D2D chunks,
    # STAGE for 256 MiB of D2D chunks whose phases differ; the tail policy keeps its 4 bulk CTAs
    s = (1 << 32) + 32768 * g.permutation(32768)[:16384].astype(np.uint64)
    d = (1 << 36) + 32768 * np.arange(16384, dtype=np.uint64)
    z = np.full(16384, 16384, dtype=np.uint64)
    assert kvx.kvx_auto_path(s, d, z, None, "d2d") == "kernel_ldg"
    assert kvx.kvx_auto_path(s + np.uint64(8), d, z, None, "d2d") == "kernel_stage"
    assert kvx.kvx_auto_path(s + np.uint64(8), d, z, None, "d2d", "tail") == "kernel_bulk"
    assert kvx.kvx_auto_path(s + np.uint64(8), d, z, None, "h2d") == "kernel_ldg"
    with pytest.raises(kvx.KvxError):
        kvx.kvx_auto_path([1 << 30], [1 << 40], [12], None, "h2d")
    with pytest.raises(kvx.KvxError):
        kvx.kvx_auto_path([1 << 30], [1 << 40], [8], None, "h2d", 7)


def _run_with_env(code, **env_vars):
    env = dict(os.environ, **env_vars)
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)


def test_kvx_table_file_overrides_rows(tmp_path):
    table = tmp_path / "gb300.table"
    table.write_text("# dir max_mean variant budget threads unroll stages policy [assign]\n"
                     "h2d 8192 bulk 7 256 8 5 0\n"
                     "h2d inf ldg 33 512 4 3 1 static\n"
                     "d2d inf bulk 11 256 8 4 0 auto 1099511627776\n"  # batches of 1 TiB and more
                     "d2d inf ldg 99 512 8 3 0 dynamic\n"
                     "d2h inf stage 21 128 8 2 0 auto 0 unmatched\n"
                     "d2h inf ldg 13 512 8 3 0 auto 0 any 65536\n")
    code = ("from expert_host_block_gb300 import kvx\n"
            "print(kvx.kvx_default_launch('h2d', 4096))\n"
            "print(kvx.kvx_default_launch('h2d', 16384))\n"
            "print(kvx.kvx_default_launch('d2h', 4096))\n"
            "print(kvx.kvx_default_launch('d2d', 4096))\n")
    out = _run_with_env(code, KVX_TABLE=str(table))
    lines = out.stdout.strip().splitlines()
    assert "'variant': 2, 'cta_budget': 7" in lines[0] and "'stages': 5" in lines[0], out.stderr
    assert "'assign': 2" in lines[0]  # no assign column: the built-in choice for h2d
    assert "'cta_budget': 33, 'threads': 512, 'unroll': 4" in lines[1] and "'assign': 1" in lines[1]
    assert "'variant': 1, 'cta_budget': 64" in lines[2]  # no d2h row in the file: built-in row
    # kvx_default_launch describes a large batch: the 1 TiB row applies (assign auto: static for d2d)
    assert "'variant': 2, 'cta_budget': 11" in lines[3] and "'assign': 1" in lines[3]
    # the phase column: the d2h stage row applies only to batches whose phases differ
    code2 = ("import numpy as np\n"
             "from expert_host_block_gb300 import kvx\n"
             "i = np.arange(64, dtype=np.uint64)\n"
             "s = np.uint64(1 << 36) + i * np.uint64(8192)\n"
             "d = np.uint64(1 << 32) + i * np.uint64(8192)\n"
             "z = np.full(64, 4096, dtype=np.uint64)\n"
             "print(kvx.kvx_select_launch(s, d, z, None, 'd2h')['variant'])\n"
             "print(kvx.kvx_select_launch(s + np.uint64(8), d, z, None, 'd2h')['variant'])\n")
    out = _run_with_env(code2, KVX_TABLE=str(table))
    assert out.stdout.split() == ["1", "3"], out.stdout + out.stderr
    # the max_payload column: a d2h batch of at most 64 KiB takes the 512-thread row (after the stage
    # row, which it matches only with phases that differ); a bigger one the built-in 256-thread row
    code3 = ("import numpy as np\n"
             "from expert_host_block_gb300 import kvx\n"
             "i = np.arange(16, dtype=np.uint64)\n"
             "s = np.uint64(1 << 36) + i * np.uint64(8192)\n"
             "d = np.uint64(1 << 32) + i * np.uint64(8192)\n"
             "print(kvx.kvx_select_launch(s, d, np.full(16, 4096, dtype=np.uint64), None, 'd2h')['threads'])\n"
             "print(kvx.kvx_select_launch(s, d, np.full(16, 8192, dtype=np.uint64), None, 'd2h')['threads'])\n")
    out = _run_with_env(code3, KVX_TABLE=str(table))
    assert out.stdout.split() == ["512", "256"], out.stdout + out.stderr


@pytest.mark.parametrize("text", ["h2d 4096 tma 8 256 8 3 0\n", "h2d 4096 ldg 8 300 8 3 0\n",
                                  "x2y inf ldg 8 256 8 3 0\n", "h2d inf ldg 8 256 8\n",
                                  "h2d inf ldg 8 256 8 3 0 greedy\n", "h2d inf ldg 8 256 8 3 0 auto 12x\n",
                                  "d2d inf stage 8 128 8 3 0\n", "d2d inf ldg 8 256 8 3 0 auto 0 odd\n",
                                  "d2d inf ldg 8 256 8 3 0 auto 0 any 12q\n"])
def test_kvx_table_malformed_is_an_error(tmp_path, text):
    table = tmp_path / "bad.table"
    table.write_text(text)
    code = ("from expert_host_block_gb300 import kvx\n"
            "try:\n"
            "    kvx.kvx_copy_batch([8], [16], [8], None, 0, 0, None)\n"
            "except kvx.KvxError as e:\n"
            "    print(e.status, e)\n")
    out = _run_with_env(code, KVX_TABLE=str(table))
    assert out.stdout.startswith(f"{kvx.KVX_ERR_INVALID_ARG} ") and "KVX_TABLE" in out.stdout, out.stdout + out.stderr
    out = _run_with_env(code, KVX_TABLE=str(tmp_path / "missing.table"))
    assert "cannot open" in out.stdout


def test_kvx_log_reports_failures_on_stderr():
    code = ("from expert_host_block_gb300 import kvx\n"
            "print(kvx.kvx_validate([8], [16], [12], None, 0, 0))\n")
    out = _run_with_env(code, KVX_LOG="1")
    assert out.stdout.strip() == str(kvx.KVX_ERR_ALIGN)
    assert "kvx: status 2:" in out.stderr and "multiples of 8" in out.stderr
    out = _run_with_env(code, KVX_LOG="0")
    assert "kvx:" not in out.stderr
    bad = ("from expert_host_block_gb300 import kvx\n"
           "try:\n"
           "    kvx.kvx_copy_batch([8], [16], [8], None, 0, 0, None)\n"
           "except kvx.KvxError as e:\n"
           "    print(e.status, e)\n")
    out = _run_with_env(bad, KVX_LOG="9")
    assert out.stdout.startswith(f"{kvx.KVX_ERR_INVALID_ARG} ") and "KVX_LOG" in out.stdout


# ---- kvx_select_launch: the launch a batch gets, decided on the host ----------

def _batch(n, size, slot=None, src_phase=0, base_src=1 << 32, base_dst=1 << 36):
    slot = slot or size
    i = np.arange(n, dtype=np.uint64)
    return (np.uint64(base_src + src_phase) + i * np.uint64(slot), np.uint64(base_dst) + i * np.uint64(slot),
            np.full(n, size, dtype=np.uint64))


def test_select_launch_kv_burst_and_tiny():
    l = kvx.kvx_select_launch(*_batch(16384, 4096), None, "h2d")
    assert (l["variant"], l["cta_budget"], l["threads"], l["unroll"]) == (kvx.KVX_VARIANT_LDG, 64, 256, 8)
    assert l["assign"] == kvx.KVX_ASSIGN_DYNAMIC  # 16,384 units over 512 warps
    l = kvx.kvx_select_launch(*_batch(1024, 4096), None, "d2h")
    assert l["assign"] == kvx.KVX_ASSIGN_STATIC  # 2 units a warp: by position
    assert l["stages"] == 0  # not used by LDG
    l = kvx.kvx_select_launch(*_batch(3, 4096), None, "h2d")
    assert l["cta_budget"] == 1  # the grid never exceeds the work
    assert kvx.kvx_select_launch([], [], [], None, "h2d")["cta_budget"] == 0


def test_select_launch_d2d_rows_follow_payload_and_alignment(tmp_path):
    # phase-matched 16 KiB chunks: LDG with 9,728 CTAs from 256 MiB up, 3,648 below (above 48 MiB)
    big = kvx.kvx_select_launch(*_batch(16384, 16384), None, "d2d")
    assert (big["variant"], big["cta_budget"], big["threads"]) == (kvx.KVX_VARIANT_LDG, 9728, 128)
    below = kvx.kvx_select_launch(*_batch(16383, 16384), None, "d2d")
    assert (below["variant"], below["cta_budget"], below["threads"]) == (kvx.KVX_VARIANT_LDG, 3648, 128)
    # chunks of 16 and 8 KiB (mean 12 KiB) alike
    assert kvx.kvx_select_launch(*_batch(16384, 24576), None, "d2d")["cta_budget"] == 9728
    odd = kvx.kvx_select_launch(*_batch(4096, 16384, slot=32768, src_phase=8), None, "d2d")
    assert odd["variant"] == kvx.KVX_VARIANT_LDG  # 64 MiB with phases that differ: below the STAGE row
    # a bulk row (from a table file) takes a batch with 9 % of its bytes misaligned (source and
    # destination shifted alike), not one with 11 %
    table = tmp_path / "t.txt"
    table.write_text("d2d inf bulk 456 256 8 6 0 auto 268435456\n")
    code = ("import sys, numpy as np\n"
            "sys.path.insert(0, 'tests')\n"
            "from test_abi_host import _batch\n"
            "from expert_host_block_gb300 import kvx\n"
            "s, d, z = _batch(20000, 16384, slot=32768)\n"
            "s[:1800] += 8; d[:1800] += 8\n"
            "a = kvx.kvx_select_launch(s, d, z, None, 'd2d')['variant']\n"
            "s[:2200] = s[:2200] | 8; d[:2200] = d[:2200] | 8\n"
            "b = kvx.kvx_select_launch(s, d, z, None, 'd2d')['variant']\n"
            "print(a, b)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=root,
                         env=dict(os.environ, KVX_TABLE=str(table)))
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(kvx.KVX_VARIANT_BULK), str(kvx.KVX_VARIANT_LDG)]
    # small chunks stay with LDG at any payload
    assert kvx.kvx_select_launch(*_batch(65536, 4096), None, "d2d")["variant"] == kvx.KVX_VARIANT_LDG
    # an explicit request wins over the table
    forced = kvx.kvx_select_launch(*_batch(64, 16384, slot=32768, src_phase=8), None, "d2d", {"variant": "bulk"})
    assert forced["variant"] == kvx.KVX_VARIANT_BULK
    forced = kvx.kvx_select_launch(*_batch(16384, 4096), None, "h2d", {"assign": "static", "cta_budget": 7})
    assert forced["assign"] == kvx.KVX_ASSIGN_STATIC and forced["cta_budget"] == 7


def test_select_launch_stage_row_for_mismatched_phases():
    # D2D batches of 128 MiB or more with a chunk whose source and destination differ mod 16
    l = kvx.kvx_select_launch(*_batch(65536, 4096, slot=8192, src_phase=8), None, "d2d")
    assert (l["variant"], l["threads"], l["unroll"], l["stages"]) == (kvx.KVX_VARIANT_STAGE, 128, 0, 2)
    assert l["cta_budget"] == 2432 and l["assign"] == 0  # chunks of one 4 KiB unit: 2 stages, 2,432 CTAs
    l = kvx.kvx_select_launch(*_batch(32768, 8192, slot=16384, src_phase=8), None, "d2d")
    assert (l["variant"], l["stages"], l["cta_budget"]) == (kvx.KVX_VARIANT_STAGE, 4, 3648)  # longer chunks
    # one mismatched chunk is enough; 16-byte phases that agree are not
    s, d, z = _batch(32768, 8192, slot=16384)
    assert kvx.kvx_select_launch(s, d, z, None, "d2d")["variant"] == kvx.KVX_VARIANT_LDG
    s[7] += 8
    assert kvx.kvx_select_launch(s, d, z, None, "d2d")["variant"] == kvx.KVX_VARIANT_STAGE
    # below 128 MiB, and over the host link, LDG
    assert kvx.kvx_select_launch(*_batch(16383, 8192, slot=16384, src_phase=8), None,
                                 "d2d")["variant"] == kvx.KVX_VARIANT_LDG
    assert kvx.kvx_select_launch(*_batch(65536, 4096, slot=8192, src_phase=8), None,
                                 "h2d")["variant"] == kvx.KVX_VARIANT_LDG
    # asked for: the grid follows 4 warps a CTA, one 4 KiB unit each per pass; stages 2, 4 or 8 only
    l = kvx.kvx_select_launch(*_batch(100, 16384), None, "h2d", {"variant": "stage", "stages": 8, "cta_budget": 999})
    assert (l["variant"], l["cta_budget"], l["stages"]) == (kvx.KVX_VARIANT_STAGE, 100, 8)
    l = kvx.kvx_select_launch(*_batch(100, 16384), None, "h2d", {"variant": "stage"})
    assert l["stages"] == 4  # the h2d row's stages belong to another variant
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_select_launch(*_batch(100, 16384), None, "h2d", {"variant": "stage", "stages": 3})
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG


def test_select_launch_small_d2d_row():
    # D2D batches of at most 24 MiB: one 512-thread CTA per SM; from just above it, 128-thread CTAs:
    # for phase-matched batches 1,824 of them up to 48 MiB and 3,648 above; for batches with a chunk
    # whose phases differ (the one-path instance) 1,216 up to 32 MiB and 3,040 above, up to the STAGE
    # row's 128 MiB
    small = kvx.kvx_select_launch(*_batch(6144, 4096), None, "d2d")  # 24 MiB
    assert (small["variant"], small["threads"], small["unroll"]) == (kvx.KVX_VARIANT_LDG, 512, 8)
    assert small["cta_budget"] == 152  # 6,144 units need 384 CTAs of 16 warps: the budget binds
    assert kvx.kvx_select_launch(*_batch(1024, 4096), None, "d2d")["cta_budget"] == 64  # 1,024 units: the work binds
    big = kvx.kvx_select_launch(*_batch(6146, 4096), None, "d2d")
    assert (big["threads"], big["cta_budget"]) == (128, 1537)  # 6,146 units of 4 warps a CTA: the work binds
    assert kvx.kvx_select_launch(*_batch(16384, 4096), None, "d2d")["cta_budget"] == 3648  # 64 MiB, matched
    assert kvx.kvx_select_launch(*_batch(12288, 4096), None, "d2d")["cta_budget"] == 1824  # 48 MiB, matched
    odd = kvx.kvx_select_launch(*_batch(16384, 4096, slot=8192, src_phase=8), None, "d2d")  # 64 MiB, mismatched
    assert (odd["variant"], odd["threads"], odd["cta_budget"]) == (kvx.KVX_VARIANT_LDG, 128, 3040)
    odd = kvx.kvx_select_launch(*_batch(7168, 4096, slot=8192, src_phase=8), None, "d2d")  # 28 MiB, mismatched
    assert (odd["threads"], odd["cta_budget"]) == (128, 1216)
    # host-link batches of any size keep their row
    assert kvx.kvx_select_launch(*_batch(4096, 4096), None, "h2d")["threads"] == 256


def test_select_launch_rejects_what_copy_batch_rejects():
    s, d, z = _batch(4, 4096)
    z[2] = 12
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_select_launch(s, d, z, None, "h2d")
    assert e.value.status == kvx.KVX_ERR_ALIGN
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_select_launch(*_batch(4, 4096), None, 9)
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG


def test_select_launch_with_table_file_payload_rows(tmp_path):
    table = tmp_path / "rows.table"
    table.write_text("d2d inf ldg 77 128 4 3 0 static 2147483648\n")  # batches of 2 GiB and more
    code = ("import numpy as np\n"
            "from expert_host_block_gb300 import kvx\n"
            "for n in (2, 1):\n"
            "    s = np.uint64(1 << 32) + np.arange(n, dtype=np.uint64) * np.uint64(1 << 31)\n"
            "    d = np.uint64(1 << 40) + np.arange(n, dtype=np.uint64) * np.uint64(1 << 31)\n"
            "    z = np.full(n, 1 << 30, dtype=np.uint64)\n"
            "    print(kvx.kvx_select_launch(s, d, z, None, 'd2d'))\n")
    out = _run_with_env(code, KVX_TABLE=str(table))
    lines = out.stdout.strip().splitlines()
    assert "'cta_budget': 77, 'threads': 128, 'unroll': 4" in lines[0], out.stderr
    assert "'variant': 1, 'cta_budget': 9728" in lines[1]  # 1 GiB: the file row does not apply, the built-in one does


def test_nvtx_switch_accepted():
    # KVX_NVTX=1 only adds profiler ranges; host-only entry points behave the same
    code = ("from expert_host_block_gb300 import kvx\n"
            "print(kvx.kvx_select_launch([8], [16], [8], None, 'h2d')['variant'])\n"
            "print(kvx.kvx_validate([8], [16], [12], None, 0, 0))\n")
    for v in ("0", "1"):
        out = _run_with_env(code, KVX_NVTX=v)
        assert out.returncode == 0, out.stderr
        assert out.stdout.split() == [str(kvx.KVX_VARIANT_LDG), str(kvx.KVX_ERR_ALIGN)]


def test_debug_bounds_argument_errors_need_no_device():
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_debug_bounds(np.arange(65, dtype=np.uint64) << np.uint64(20),
                             (np.arange(65, dtype=np.uint64) + np.uint64(1)) << np.uint64(20))
    assert e.value.status == kvx.KVX_ERR_CAPACITY
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_debug_bounds([4096, 1 << 20], [8192, 1 << 19])  # the second range is reversed
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        kvx.kvx_debug_bounds([4096], [])


def test_stale_and_bogus_handles_are_argument_errors():
    # A destroyed handle, a pointer that never was a handle, or a handle of another
    # kind is rejected before the library touches it (no device needed).
    lib = kvx._load()
    t = kvx.Transfer()
    stale = t.handle
    t.close()
    done = ctypes.c_int()
    assert lib.kvx_transfer_poll(stale, ctypes.byref(done)) == kvx.KVX_ERR_INVALID_ARG
    assert lib.kvx_transfer_progress(stale, None, None) == kvx.KVX_ERR_INVALID_ARG
    assert lib.kvx_transfer_destroy(stale) == kvx.KVX_ERR_INVALID_ARG  # destroyed twice
    assert "not a live transfer" in kvx.last_error()
    with pytest.raises(kvx.KvxError) as e:
        kvx.Transfer.start(types.SimpleNamespace(handle=stale), [8], [16], [8], "h2d")
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG

    bogus = ctypes.create_string_buffer(4096)
    addr = ctypes.addressof(bogus)
    live = kvx.Transfer()  # a live handle of the wrong kind
    try:
        for h in (addr, live.handle):
            for call in (lambda: kvx.kvx_desc_buf_info(h),
                         lambda: kvx.kvx_copy_uploaded(h),
                         lambda: kvx.kvx_upload_descriptors(h, [8], [16], [8], None, "h2d"),
                         lambda: kvx.kvx_desc_buf_destroy(h),
                         lambda: kvx.kvx_devlist_destroy(h),
                         lambda: kvx.kvx_copy_device_list(h, 8, 8, 8, 4, "d2d")):
                with pytest.raises(kvx.KvxError) as e:
                    call()
                assert e.value.status == kvx.KVX_ERR_INVALID_ARG and "not a live" in str(e.value)
        assert bytes(bogus.raw) == bytes(4096)  # never written
        assert live.progress() == (0, 0)  # the live transfer is untouched
    finally:
        live.close()
