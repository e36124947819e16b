"""CPU checks of the host-side logic of pipeline.py: the packed step I/O layout."""
import torch

from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch, logits_ld


def test_packed_io_views_alias_one_buffer_at_aligned_offsets():
    ts = [torch.randn(3, 5, 7).to(torch.bfloat16), torch.randn(3, 64), torch.arange(5, dtype=torch.int64),
          torch.arange(9, dtype=torch.int32).view(3, 3)]
    buf, views = DeviceBatch._packed(ts, "cpu")
    base = buf.data_ptr()
    end = 0
    for t, v in zip(ts, views):
        off = v.data_ptr() - base
        assert off % 256 == 0 and off >= end                  # aligned, in order, no overlap
        end = off + v.numel() * v.element_size()
        assert v.shape == t.shape and v.dtype == t.dtype and v.is_contiguous()
        v.copy_(t)
    assert end <= buf.numel()
    for t, v in zip(ts, views):                               # the data lives in the one buffer
        assert torch.equal(v, t)
    # bytes between the tensors (padding) stay zero
    covered = torch.zeros(buf.numel(), dtype=torch.bool)
    for v in views:
        o = v.data_ptr() - base
        covered[o:o + v.numel() * v.element_size()] = True
    assert int(buf[~covered].abs().sum()) == 0


def test_logits_row_stride_is_16_byte_rounded():
    assert logits_ld(1) == 4 and logits_ld(4) == 4 and logits_ld(5) == 8 and logits_ld(65536) == 65536
