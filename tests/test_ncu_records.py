"""The committed ncu records (DRAM bytes, tensor-pipe activity) and the digest
that ties each to the kernel source it was taken on.  The digest covers the
code lines alone: a comment edit keeps a record valid, any change to the code
makes bench.py report null for it."""
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // one\n'
           'const char *s = "// not a comment /* nor this */";\n'
           '/* block\n   over two lines */ int b = \'/\';\n'
           'char q = \'"\'; int c = 2; /**/ int d = 3;\n')
    out = bench.strip_comments(src)
    assert out.splitlines() == ['int a = 1; ',
                                'const char *s = "// not a comment /* nor this */";',
                                '',
                                ' int b = \'/\';',
                                'char q = \'"\'; int c = 2;  int d = 3;']


def _copy_sources(tmp_path):
    dst = tmp_path / "io_aware_exact_09_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "io_aware_exact_09_gb300", "csrc"), dst,
                    ignore=shutil.ignore_patterns("*.so", "*.o", "_build*"))
    return dst


def test_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    name = bench.KERNEL_SOURCES["fa_fwd_kernel"]
    name = name if isinstance(name, str) else sorted(name)[0]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.source_digest(name)
    f = dst / name
    text = f.read_text()
    f.write_text("// an added comment line\n\n" + text.replace("\n", "   \n", 1) + "/* trailing */\n")
    assert bench.source_digest(name) == before
    f.write_text(text + "static int fa_extra_symbol = 0;\n")
    assert bench.source_digest(name) != before
    # the shared device headers count for every kernel
    f.write_text(text)
    h = dst / "fa_tiles.cuh"
    h.write_text(h.read_text() + "struct FaExtra {};\n")
    assert bench.source_digest(name) != before


def test_records_are_current_and_complete():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as fh:
        rows = json.load(fh)
    seen = 0
    for kernel, by_workload in rows.items():
        if kernel.startswith("_"):
            continue
        assert kernel in bench.KERNEL_SOURCES, kernel
        for workload, r in by_workload.items():
            assert r["source_digest"] == bench.source_digest(bench.KERNEL_SOURCES[kernel]), (kernel, workload)
            assert r["bytes_per_launch"] == r["read"] + r["write"] > 0, (kernel, workload)
            assert "--clock-control none" in r["command"], (kernel, workload)
            seen += 1
    assert seen >= 10
