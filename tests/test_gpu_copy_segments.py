"""pa_copy_segments: several copies in one kernel, the segment list read when the kernel runs
(page-locked host memory), so a captured graph follows a rewritten list."""

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _segments(pa, triples):
    buf = torch.zeros(max(len(triples), 1) * ctypes.sizeof(pa.CopySegment), dtype=torch.uint8).pin_memory()
    segs = (pa.CopySegment * max(len(triples), 1)).from_address(buf.data_ptr())
    for i, (src, dst, n) in enumerate(triples):
        segs[i].src, segs[i].dst, segs[i].bytes = src, dst, n
    return buf, segs


def test_copy_segments_every_alignment_and_direction(pa):
    gen = torch.Generator().manual_seed(200)
    host = torch.randint(0, 256, (1 << 20,), dtype=torch.uint8, generator=gen).pin_memory()
    dev = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    back = torch.zeros(1 << 20, dtype=torch.uint8).pin_memory()
    # (source offset, destination offset, bytes): aligned, odd sizes, misaligned either side, empty
    cases = [(0, 0, 1 << 18), (16, 300032, 4093), (3, 400000, 70001), (4096, 500001, 5), (0, 600000, 0),
             (7, 700003, 65536)]
    buf, _ = _segments(pa, [(host.data_ptr() + s, dev.data_ptr() + d, n) for s, d, n in cases])
    pa.copy_segments(buf.data_ptr(), len(cases))
    buf2, _ = _segments(pa, [(dev.data_ptr() + d, back.data_ptr() + d, n) for s, d, n in cases])
    pa.copy_segments(buf2.data_ptr(), len(cases))
    torch.cuda.synchronize()
    d = dev.cpu()
    for s, o, n in cases:
        assert torch.equal(d[o:o + n], host[s:s + n]), (s, o, n)
        assert torch.equal(back[o:o + n], host[s:s + n]), (s, o, n)
    # bytes outside the segments untouched
    assert int(d[1 << 18:300032].abs().sum()) == 0


def test_copy_segments_in_a_graph_follows_the_rewritten_list(pa):
    a = torch.arange(4096, dtype=torch.int32).pin_memory()
    b = (torch.arange(4096, dtype=torch.int32) * 7).pin_memory()
    dst = torch.zeros(4096, dtype=torch.int32, device="cuda")
    buf, segs = _segments(pa, [(a.data_ptr(), dst.data_ptr(), a.numel() * 4)])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.copy_segments(buf.data_ptr(), 1)  # warm-up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.copy_segments(buf.data_ptr(), 1)
    torch.cuda.synchronize()
    for src in (b, a, b):
        segs[0].src = src.data_ptr()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dst.cpu(), src)


def test_copy_segments_argument_checks(pa):
    lib = pa.library()
    assert lib.pa_copy_segments(None, 0, None) == 0
    assert lib.pa_copy_segments(None, 1, None) == -1
    buf, _ = _segments(pa, [])
    assert lib.pa_copy_segments(ctypes.c_void_p(buf.data_ptr()), 65, None) == -1
    assert lib.pa_copy_segments(ctypes.c_void_p(buf.data_ptr()), -1, None) == -1
