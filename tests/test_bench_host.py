"""Host-side helpers of bench.py that need no GPU: the packed input staging
used by the end-to-end measurements, and the hash that ties the reported
DRAM traffic to the decode sources it was measured on."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture
def no_pinning(monkeypatch):
    """Pinned host memory needs a CUDA driver; the layout logic does not."""
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)


def test_host_stage_round_trip_and_alignment(no_pinning):
    g = torch.Generator().manual_seed(0)
    parts = {
        "q": torch.randn(3, 5, 7, generator=g).to(torch.bfloat16),
        "bt": torch.arange(33, dtype=torch.int32).view(3, 11),
        "lens": torch.tensor([7, 8, 9], dtype=torch.int32),
        "k_new": torch.randn(3, 1, 2, 4, generator=g),
        "slots": torch.tensor([5, 600, 70001], dtype=torch.int64),
        "one_byte": torch.tensor([1], dtype=torch.uint8),
    }
    st = bench._HostStage(parts)
    offsets = [o for _, o, _, _, _ in st.layout]
    assert all(o % 256 == 0 for o in offsets)
    assert offsets == sorted(offsets) and len(set(offsets)) == len(offsets)
    assert st.nbytes % 256 == 0 and st.nbytes >= sum(t.numel() * t.element_size() for t in parts.values())
    views = st.upload("cpu")
    assert list(views) == list(parts)
    for name, t in parts.items():
        assert views[name].dtype == t.dtype and views[name].shape == t.shape
        assert torch.equal(views[name], t)


def test_host_stage_views_are_persistent_and_refreshed(no_pinning):
    parts = {"a": torch.zeros(4, dtype=torch.float32), "b": torch.ones(2, 2, dtype=torch.int32)}
    st = bench._HostStage(parts)
    v1 = st.upload("cpu")
    # a new step's inputs written into the pinned buffer reach the same views
    st.buf[0:16].copy_(torch.arange(4, dtype=torch.float32).view(torch.uint8))
    v2 = st.upload("cpu")
    assert v2["a"].data_ptr() == v1["a"].data_ptr()
    assert torch.equal(v2["a"], torch.arange(4, dtype=torch.float32))
    assert torch.equal(v2["b"], torch.ones(2, 2, dtype=torch.int32))


def test_host_stage_non_contiguous_input(no_pinning):
    t = torch.arange(24, dtype=torch.float32).view(4, 6).t()      # a transposed view
    st = bench._HostStage({"t": t})
    assert torch.equal(st.upload("cpu")["t"], t.contiguous())


def test_kernel_hash_ignores_comments_but_not_code():
    """The DRAM traffic bench.py reports is tied to the decode sources the
    ncu counters were taken on: comments and blank lines may change without
    invalidating it, any code token may not."""
    src = (
        "// header comment\n"
        "#include \"internal.h\"\n"
        "/* a block\n   comment */\n"
        "__global__ void k(int *p)   // trailing\n"
        "{\n"
        "\n"
        "    p[0] = 1;   /* inline */ p[1] = 2;\n"
        "}\n"
    )
    base = bench._code_only(src)
    assert "comment" not in base and "trailing" not in base and "inline" not in base
    assert bench._code_only(src.replace("// header comment", "// another header")) == base
    assert bench._code_only(src.replace("\n\n", "\n\n\n\n")) == base
    assert bench._code_only(src.replace("p[1] = 2", "p[1] = 3")) != base
    assert bench._code_only(src.replace("p[0]", "p [0]")) != base
    # the committed traffic table is keyed by this hash of the current sources
    assert len(bench._kernel_sha()) == 16
