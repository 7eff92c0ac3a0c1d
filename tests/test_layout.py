"""CPU checks of the tiled cache-page layout helpers (8x8 core matrices per page and head)."""
import torch

from invariant_hybrid_attention_gb300.paged import tile, tile_v256, untile, untile_rot, untile_v256


def test_tile_untile_roundtrip():
    x = torch.arange(3 * 2 * 16 * 256, dtype=torch.float32).view(3, 2, 16, 256)
    t = tile(x)
    assert t.shape == (3, 2, 2, 32, 8, 8)
    # key j, dim d sits at ((j // 8) * (D // 8) + d // 8) * 64 + (j % 8) * 8 + d % 8 of a block
    flat = t.reshape(3, 2, -1)
    for j, d in [(0, 0), (5, 9), (8, 7), (15, 255), (9, 130)]:
        assert flat[1, 1, ((j // 8) * 32 + d // 8) * 64 + (j % 8) * 8 + d % 8] == x[1, 1, j, d]
    assert torch.equal(untile(t), x)


def test_global_half_layout_roundtrip():
    x = torch.arange(2 * 3 * 16 * 512, dtype=torch.float32).view(2, 3, 16, 512)
    t = tile(x)
    assert t.shape == (2, 3, 2, 2, 32, 8, 8)
    flat = t.reshape(2, 3, -1)
    # key j, dim d at (((d // 256) * 2 + j // 8) * 32 + (d % 256) // 8) * 64 + (j % 8) * 8 + d % 8
    for j, d in [(0, 0), (5, 9), (8, 263), (15, 511), (9, 300), (3, 255)]:
        off = (((d // 256) * 2 + j // 8) * 32 + (d % 256) // 8) * 64 + (j % 8) * 8 + d % 8
        assert flat[1, 2, off] == x[1, 2, j, d]
    assert torch.equal(untile(t), x)
    # each 256-dim half of a page-head is one contiguous 4096-element block
    assert torch.equal(flat[0, 0, 4096:8192].sort().values, x[0, 0, :, 256:].reshape(-1).sort().values)


def test_rotated_side_layout():
    # element of key j, rotated dim d (d in [0,64) or [256,320)):
    #   (((d // 256) * 2 + j // 8) * 8 + (d % 64) // 8) * 64 + (j % 8) * 8 + d % 8
    t = torch.arange(2 * 4 * 2048, dtype=torch.float32).view(2, 4, 2, 2, 8, 8, 8)
    rows = untile_rot(t)
    assert rows.shape == (2, 4, 16, 128)
    flat = t.reshape(2, 4, -1)
    for j, d in [(0, 0), (7, 63), (8, 256), (15, 319), (10, 300)]:
        col = d if d < 64 else d - 256 + 64
        off = (((d // 256) * 2 + j // 8) * 8 + (d % 64) // 8) * 64 + (j % 8) * 8 + d % 8
        assert rows[1, 3, j, col] == flat[1, 3, off]


def test_sliding_v_half_layout_roundtrip():
    # sliding V: key j, dim d at (((d // 128) * 2 + j // 8) * 16 + (d % 128) // 8) * 64 + (j % 8) * 8 + d % 8
    x = torch.arange(3 * 2 * 16 * 256, dtype=torch.float32).view(3, 2, 16, 256)
    t = tile_v256(x)
    assert t.shape == (3, 2, 2, 2, 16, 8, 8)
    flat = t.reshape(3, 2, -1)
    for j, d in [(0, 0), (5, 9), (8, 127), (15, 255), (9, 130), (3, 128)]:
        off = (((d // 128) * 2 + j // 8) * 16 + (d % 128) // 8) * 64 + (j % 8) * 8 + d % 8
        assert flat[2, 1, off] == x[2, 1, j, d]
    assert torch.equal(untile_v256(t), x)
    # each 128-dim half of a page-head block is one contiguous 2048-element (4 KB) block
    assert torch.equal(flat[0, 0, 2048:].sort().values, x[0, 0, :, 128:].reshape(-1).sort().values)
