"""The committed Nsight Compute summaries describe the kernels as they are:
each names the sha256 of the kernel source it was captured on, and that
must be the source's current hash (a changed kernel needs a new capture).
Older hashes may still be quoted for comparison; the current one must be
among them."""
import hashlib
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "roofline_driven_optimisation_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")

# summary -> kernel sources whose counters it reports
SOURCES = {
    "attention_kernel_causal_2048.md": ["attention.cu"],
    "attention_kernel_noncausal_4096.md": ["attention.cu"],
    "gemm_bf16_tc2_kernel_bf16_8192.md": ["gemm_bf16_tc2.cu"],
    "gemm_bf16_tc2_kernel_fp8_e4m3_4096.md": ["gemm_bf16_tc2.cu"],
    "gemm_bf16_tc2_kernel_swiglu_prefill_m2048.md": ["gemm_bf16_tc2.cu"],
    "gemm_bf16_tc_kernel_bf16_8192.md": ["gemm_bf16_tc.cu"],
    "gemm_skinny_kernel_decode_split_choice.md": ["gemm_skinny.cu"],
    "gemm_skinny_kernel_swiglu_decode_m16.md": ["gemm_skinny.cu"],
    "gemm_w4_decode_kernel_lm_m16.md": ["gemm_w4_decode.cu"],
    "int4_dequant_bf16_16384.md": ["int4_dequant.cu"],
    "launch_list_bench_step.md": ["gemm_f32_simt.cu", "gemm_skinny.cu", "gemm_bf16_tc2.cu"],
    "sgemm_tma_kernel_fp32_4096.md": ["gemm_f32_simt.cu"],
}


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def test_every_summary_is_listed():
    on_disk = {f for f in os.listdir(PROFILES) if f.endswith(".md") and f != "README.md"}
    assert on_disk == set(SOURCES), sorted(on_disk ^ set(SOURCES))


@pytest.mark.parametrize("summary", sorted(SOURCES))
def test_summary_names_current_source_hash(summary):
    with open(os.path.join(PROFILES, summary), encoding="utf-8") as f:
        text = f.read()
    for src in SOURCES[summary]:
        h = _sha(os.path.join(CSRC, src))
        assert h in text, f"{summary} was captured on another {src} (current sha256 {h})"

