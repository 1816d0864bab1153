"""The benchmark's host logic that needs no GPU: which projection kernel a
workload's roofline covers, and when a committed ncu summary still applies
(its recorded hash of that kernel's source files must match the sources)."""
import os

import bench


def test_projection_kernel_per_workload():
    assert bench.projection_kernel("pr1", 1) == "head_gemm_kernel"
    assert bench.projection_kernel("pr1", 512) == "head_gemm_kernel"     # --batch: int8 only
    assert bench.projection_kernel("sweep", 512) == "head_gemm_kernel"
    assert bench.projection_kernel("spec", 256) == "head_pair_kernel"
    assert bench.projection_kernel("verify", 256) == "head_pair_kernel"
    assert bench.projection_kernel("gated", 1) == "head_gemm_kernel"
    assert bench.projection_kernel("logprob", 8192) == "head_rows_kernel"
    assert bench.projection_kernel("int8", 1) == "int8_gemm_kernel"
    assert bench.projection_kernel("int8", 512) == "head_pair_kernel"   # fp16 copies, wide path
    for kernel in {bench.projection_kernel(w, b) for w in bench.WORKLOADS for b in (1, 512)}:
        assert kernel in bench.KERNEL_SOURCES


def test_source_hash_ignores_comments_and_blank_lines():
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    assert bench._code_only(code) == bench._code_only(
        "/* a block\n comment */\nint f(int x) {\n\n  return x + 1;\n}\n")
    assert bench._code_only(code) != bench._code_only(code.replace("+ 1", "+ 2"))


def test_source_hash_covers_the_kernel_files_only():
    src = os.path.join(bench.ROOT, "invariant_output_head_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(src, f)), (kernel, f)
        h = bench.kernel_source_hash(kernel)
        assert len(h) == 16 and h == bench.kernel_source_hash(kernel)
    assert (bench.kernel_source_hash("head_gemm_kernel")
            != bench.kernel_source_hash("head_rows_kernel"))


def test_profiled_traffic_needs_a_matching_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "invariant_output_head_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["head_rows_kernel"]:
        (src / f).write_text(f"// {f}\nint v_{f.replace('.', '_')} = 1;\n")
    assert bench.profiled_traffic("logprob", 8192) is None        # no summary yet
    good = bench.kernel_source_hash("head_rows_kernel")
    (prof / "head_rows_logprob.md").write_text(
        f"# summary\n\n- kernel_source_sha256_16: `{good}`\n- dram_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic("logprob", 8192) == 12345.0
    # a comment change keeps the summary, a code change retires it
    (src / "rows_kernels.cuh").write_text("// reworded\nint v_rows_kernels_cuh = 1;\n")
    assert bench.profiled_traffic("logprob", 8192) == 12345.0
    (src / "rows_kernels.cuh").write_text("int v_rows_kernels_cuh = 2;\n")
    assert bench.profiled_traffic("logprob", 8192) is None
