"""The key under which the bench looks up a kernel's measured DRAM traffic:
a hash of the sources that kernel is built from (its translation units,
the launch setup in api.cu and every header), so a capture stays valid while
those files are unchanged and is dropped as soon as one of them changes."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

CSRC = os.path.join(ROOT, "moe_mx8_quantize_gb300", "csrc")
STEP_LABELS = [lab for branch in bench.Step.BRANCHES for lab in branch]


def _tus(label):
    return next((t for prefix, t in bench.KERNEL_TUS if label.startswith(prefix)), None)


def test_every_step_label_has_its_translation_units():
    names = set(os.listdir(CSRC))
    for lab in STEP_LABELS:
        tus = _tus(lab)
        assert tus is not None, lab
        assert set(tus) <= names, (lab, tus)


def test_label_hash_follows_only_its_sources():
    names = sorted(os.listdir(CSRC))
    files = {n: open(os.path.join(CSRC, n), "rb").read() for n in names}

    def hash_with(label, changed):
        return bench.kernel_source_hash(label, names,
                                        lambda n: files[n] + (b" " if n == changed else b""))

    for lab in ("nvfp4_quant_expert W_gu", "mxfp8_gemm Fprop", "moe_combine", "mxfp8_quant_rc W"):
        base = hash_with(lab, None)
        assert base == bench.kernel_source_hash(lab)
        own = set(_tus(lab))
        for n in names:
            follows = n in own or n == "api.cu" or n.endswith((".cuh", ".h"))
            assert (hash_with(lab, n) != base) == follows, (lab, n)
    # no label: every file counts
    for n in names:
        assert hash_with(None, n) != hash_with(None, None)
