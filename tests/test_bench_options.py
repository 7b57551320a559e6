"""bench.py's variant options (CPU): what they accept and refuse."""

import pytest

import bench


@pytest.mark.parametrize("argv", [
    ["--mask", "per_head", "--impl", "reference"],
    ["--fp8", "--impl", "reference"],
    ["--mask", "shared", "--workload", "decode_b8_h32_nq1_nk32768_d128"],
    ["--fp8", "--workload", "decode_b8_h32_nq1_nk32768_d128"],
    ["--fp8", "--mask", "key_row"],
    ["--graph"],
    ["--graph", "--impl", "reference", "--workload", "single_head_n256_d64"],
    ["--splitkv"],                                          # a forward+backward workload
    ["--splitkv", "--impl", "reference", "--workload", "memory_exercise_n4096_d64"],
    ["--splitkv", "--fp8", "--workload", "memory_exercise_n4096_d64"],
    ["--bwd", "single", "--impl", "reference"],
    ["--bwd", "single", "--mask", "per_head"],
    ["--bwd", "single", "--fwd-only"],
    ["--bwd", "single", "--workload", "memory_exercise_n4096_d64"],
])
def test_variant_options_refused_where_they_do_not_apply(argv):
    with pytest.raises(SystemExit) as e:
        bench.main(argv)
    assert "appl" in str(e.value) or "no mask" in str(e.value)


def test_mask_shapes_and_defaults():
    args = bench.parse_args([])
    assert args.mask == "none" and not args.fp8
    assert set(bench.MASKS) == {"none", "key_row", "shared", "per_head"}
    assert bench.make_mask("none", 2, 3, 16, "cpu", 0) is None
    m = bench.make_mask("key_row", 2, 3, 16, "cpu", 0)
    assert tuple(m.shape) == (2, 1, 1, 16) and str(m.dtype) == "torch.bfloat16"
    assert tuple(bench.make_mask("shared", 2, 3, 16, "cpu", 0).shape) == (1, 1, 16, 16)
    assert tuple(bench.make_mask("per_head", 2, 3, 16, "cpu", 0).shape) == (1, 3, 16, 16)
    assert "fwd_fp8_kernel" in bench.KERNEL_SOURCES


def test_backward_and_split_options_defaults():
    args = bench.parse_args([])
    assert args.bwd == "two" and not args.splitkv
    for k in ("rowterm_kernel", "dkdv_kernel_dq"):
        assert k in bench.KERNEL_SOURCES
