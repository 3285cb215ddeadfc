"""Host-side helpers of bench.py: which timed steps carry per-kernel events,
and the digest that ties a measured ncu traffic figure to the kernel it was
taken from."""
import os
import shutil

import bench


def test_breakdown_steps_split_the_timed_steps():
    inner, plain = bench.breakdown_steps(2000)
    assert len(inner) == 2000 // bench.BREAKDOWN_EVERY
    assert not set(inner) & set(plain) and sorted(inner + plain) == list(range(2000))
    assert all(k % bench.BREAKDOWN_EVERY == bench.BREAKDOWN_EVERY - 1 for k in inner)
    # too few steps for a breakdown step of their own: the last one carries it,
    # and a single step serves both
    assert bench.breakdown_steps(3) == ([2], [0, 1])
    assert bench.breakdown_steps(1) == ([0], [0])


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "mla_decode_attention_03_gb300", "csrc")
    dst = tmp_path / "mla_decode_attention_03_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in {f for files in bench.KERNEL_SOURCES.values() for f in files}:
        shutil.copy(os.path.join(src, name), dst / name)
    return dst


def test_kernel_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    base = bench.kernel_digest()
    small = bench.kernel_digest("mla_decode_small_kernel")
    assert small != base
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_digest() == base
    f = dst / bench.KERNEL_SOURCES["mla_decode_kernel"][0]
    text = f.read_text(encoding="utf-8")
    f.write_text("// an added comment line\n" + text.replace("\n", "\n  ", 3), encoding="utf-8")
    assert bench.kernel_digest() == base  # comments and whitespace only
    assert "kStages = 5" in text
    f.write_text(text.replace("kStages = 5", "kStages = 4", 1), encoding="utf-8")
    assert bench.kernel_digest() != base  # a code change
    assert bench.kernel_digest("mla_decode_small_kernel") == small  # in the other kernel's file


def test_decode_kernel_by_tile_rows():
    assert bench.decode_kernel(1, 128, 1) == "mla_decode_kernel"
    assert bench.decode_kernel(2, 128, 1) == "mla_decode_kernel"
    assert bench.decode_kernel(1, 16, 1) == "mla_decode_small_kernel"
    assert bench.decode_kernel(2, 16, 2) == "mla_decode_small_kernel"   # 2 positions x 8 heads
    assert bench.decode_kernel(2, 16, 1) == "mla_decode_kernel"         # 32 rows
    assert bench.decode_kernel(1, 32, 1) == "mla_decode_kernel"


def test_passes_per_step_make_the_timed_loop_last():
    # 20 steps of 0.18 ms need 278 passes each to reach one second
    assert bench.passes_per_step(20, 0.18e-3, 1.0) == 278
    assert 20 * 278 * 0.18e-3 >= 1.0 > 20 * 277 * 0.18e-3
    # steps that already last long enough run one pass each
    assert bench.passes_per_step(20000, 0.18e-3, 1.0) == 1
    assert bench.passes_per_step(1, 5.0, 1.0) == 1
