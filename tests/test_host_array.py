"""Host-side checks of the huge-page host history array (no GPU): contents survive a remap with
MADV_COLLAPSE, and the huge fraction is reported from /proc/self/smaps."""
import pytest

torch = pytest.importorskip("torch")


def test_recollapse_keeps_contents():
    import sparse_kv_cache_decode_gb300 as K
    a = K.HostArray((1 << 28,))                   # 512 MiB of int16
    flat = a.tensor
    idx = torch.arange(0, flat.numel(), 65536)
    flat[idx] = (idx // 65536).to(torch.int16)
    before = a.huge_fraction()
    assert 0.0 <= before <= 1.0
    after = a.recollapse()                        # not registered: only the remap
    assert 0.0 <= after <= 1.0
    assert torch.equal(flat[idx], (idx // 65536).to(torch.int16))
    a.close()
