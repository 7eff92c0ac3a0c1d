"""CPU checks of the tiled cache-page layout helpers (8x8 core matrices per page and head)."""
import torch

from invariant_hybrid_attention_gb300.paged import tile, untile


def test_tile_untile_roundtrip():
    x = torch.arange(3 * 2 * 16 * 256, dtype=torch.float32).view(3, 2, 16, 256)
    t = tile(x)
    assert t.shape == (3, 2, 2, 32, 8, 8)
    # key j, dim d sits at ((j // 8) * (D // 8) + d // 8) * 64 + (j % 8) * 8 + d % 8 of a block
    flat = t.reshape(3, 2, -1)
    for j, d in [(0, 0), (5, 9), (8, 7), (15, 255), (9, 130)]:
        assert flat[1, 1, ((j // 8) * 32 + d // 8) * 64 + (j % 8) * 8 + d % 8] == x[1, 1, j, d]
    assert torch.equal(untile(t), x)
