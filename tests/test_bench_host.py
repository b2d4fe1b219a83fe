"""Host-side logic of bench.py that needs no GPU: the GEMM-source digest that
keeps measured DRAM traffic tied to the kernels it was captured on."""
import bench


def test_code_only_ignores_comments_and_keeps_code():
    a = 'int x = 1; // note\n/* block\n comment */\nint y = "//kept";\n\n'
    b = 'int x = 1;\nint y = "//kept";\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(b.replace("1", "2"))
    assert '"//kept"' in bench._code_only(a)


def test_traffic_lookup_requires_matching_workload():
    assert bench.measured_traffic("gemm_up_swiglu", "another_workload") is None
    assert bench.measured_traffic("not_a_kernel", bench.WORKLOAD) is None
