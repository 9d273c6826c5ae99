"""The bench's roofline arithmetic against the per-unit figures it is stated
in: the build's FLOPs per 64-token chunk and value head (Gram 0.524 M, W and
U 2.097 M, the two state products 4.194 M each; the first chunk of a body
skips W X), and the compose's bytes per (layer, head, segment) unit."""
import bench


def test_build_flops_per_chunk():
    d = 128
    full = 2 * 64 * 64 * d / 2 + 2 * 64 * 64 * 2 * d + 2 * (2 * 64 * d * 2 * d)
    first = full - 2 * 64 * d * 2 * d
    assert round(full) == 11_010_048 and round(first) == 6_815_744
    # the 64 x 1024-token GDN layer, 32 value heads, no seam: 16 chunks a body
    assert bench.build_flops([1024] * 64, 32) == 64 * 32 * (first + 15 * full)
    # a ragged tail of 56 tokens counts its own length
    c = 56
    tail = 2 * c * c * d / 2 + 2 * c * c * 2 * d + 2 * (2 * c * d * 2 * d)
    assert bench.build_flops([1016], 1) == first + 14 * full + tail


def test_compose_bytes_per_unit():
    L, n_seg, w, h_k, h_v = 30, 100, 8, 16, 32
    units = L * n_seg * h_v
    pair = 2 * 128 * 128 * 4
    seam_in = w * (2 * h_k * 128 * 2 + h_v * 128 * 2 + 2 * h_v * 4) / h_v  # k, q per key head; v; beta, g
    seam_out = w * 128 * 4
    states = L * h_v * 128 * 128 * 4 / units
    slots = L * n_seg * 4 / units
    assert seam_in == 4160 and seam_out == 4096
    per_unit = pair + seam_in + seam_out + states + slots
    assert abs(bench.compose_bytes(L, n_seg, w, h_k, h_v) / units - per_unit) < 1e-6
    assert bench.compose_bytes(L, n_seg, w, h_k, h_v) == 13_438_414_560
