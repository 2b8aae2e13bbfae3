"""Host-side logic of the layer helpers that needs no GPU: how StagingBuffer packs a step's
inputs (groups contiguous and in order, every tensor at a 16-byte offset, values kept) and
that it rejects groups that do not partition the staged tensors.  Pinning needs a CUDA
driver, so these tests stand the host mirror in with ordinary memory."""
import pytest
import torch

from long_context_attention_04_b300.layers import StagingBuffer


@pytest.fixture(autouse=True)
def _no_pinning(monkeypatch):
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self, *a, **k: self)


def _tensors():
    return {
        "a": torch.arange(3, dtype=torch.float32),              # 12 B -> 16
        "b": torch.arange(5, dtype=torch.int32) * 7,            # 20 B -> 32
        "c": torch.linspace(-1, 1, 7).to(torch.bfloat16),       # 14 B -> 16
        "d": torch.arange(8, dtype=torch.int64).view(2, 4),     # 64 B
    }


def test_groups_are_contiguous_aligned_and_keep_values():
    src = _tensors()
    ref = {k: v.clone() for k, v in src.items()}
    st = StagingBuffer(src, groups={"first": ["b"], "rest": ["a", "c", "d"]})
    assert st.ranges == {"first": (0, 32), "rest": (32, 32 + 16 + 16 + 64)}
    assert st.nbytes == 128
    base = st.dev_buf.data_ptr()
    for k, v in src.items():
        assert (v.data_ptr() - base) % 16 == 0
        assert v.dtype == ref[k].dtype and v.shape == ref[k].shape
        assert torch.equal(v, ref[k]) and torch.equal(st.host[k], ref[k])
    # the staged tensors are views of the packed buffer: writing the buffer changes them
    st.dev_buf.zero_()
    assert all(not v.any() for v in src.values())


def test_one_group_by_default():
    st = StagingBuffer(_tensors())
    assert st.ranges == {None: (0, st.nbytes)} and st.nbytes == 128


@pytest.mark.parametrize("groups", [{"x": ["a", "b", "c"]}, {"x": ["a", "b"], "y": ["b", "c", "d"]},
                                    {"x": ["a", "b", "c", "d", "e"]}])
def test_groups_must_partition_the_tensors(groups):
    with pytest.raises(ValueError):
        StagingBuffer(_tensors(), groups=groups)
