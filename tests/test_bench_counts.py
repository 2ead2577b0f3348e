"""The bench's algorithmic work counts (the numerators of every roofline
fraction it prints), pinned to their closed forms at the single-layer shape
B2 T2048 H16 D=N=64 Q64: 2068 bytes and 99,328 flops per token-head forward,
183,040 flops per token-head in the backward's chunk-gradient kernel."""
import bench
from state_space_sequence_complex_gb300 import inputs


def test_forward_bytes_per_token_head():
    w = inputs.LAYER
    # x, B_t, C_t read and y written at 8 B per complex value, dt read, the final state once
    assert bench.algorithmic_bytes_per_unit(w) == 16 * 64 + 16 * 64 + 4 + 8 * 64 * 64 / 2048 == 2068


def test_forward_bytes_bf16_and_real_x():
    w = inputs.LAYER
    # bfloat16 x, B_t, C_t: 768 bytes instead of 1536; a real x drops its imaginary plane
    assert bench.input_bytes_per_unit(w, bf16=True) == 2068 - 768 == 1300
    assert bench.input_bytes_per_unit(w, real_x=True) == 2068 - 256
    assert bench.input_bytes_per_unit(w, bf16=True, real_x=True) == 1300 - 128
    assert bench.input_bytes_per_unit(w) == 2068
    # the final state alone reads x (512), B_t (512) and dt (4) and writes the state once per sequence
    assert bench.input_bytes_per_unit(w, state_only=True) == 512 + 512 + 4 + 8 * 64 * 64 / 2048 == 1044
    assert bench.input_bytes_per_unit(w, state_only=True, real_x=True) == 1044 - 256


def test_forward_flops_per_token_head():
    f = bench.fp32_flops_per_unit(inputs.LAYER)
    # chunk state 8ND, state pass 8ND/Q, chunk scan over the causal triangle 4(Q+1)(N+D) + 8ND
    assert f["chunk_state"] == 8 * 64 * 64
    assert f["state_pass"] == 8 * 64 * 64 / 64
    assert f["chunk_scan"] == 4 * 65 * 128 + 8 * 64 * 64
    assert sum(f.values()) == 99328


def test_backward_flops_per_token_head():
    f = bench.bwd_flops_per_unit(inputs.LAYER)
    # per causal pair C B^T, P^H dY, dY x^H, V^T conj(C), V conj(B): 24N + 16D over (Q+1)/2 pairs,
    # plus the three state products 24ND, the row sums 16N and the chunk anchor 8ND/Q
    assert f["bwd_chunk"] == 65 * (12 * 64 + 8 * 64) + 24 * 64 * 64 + 16 * 64 + 8 * 64 * 64 / 64 == 183040
    assert f["chunk_states"] == 16 * 64 * 64
    assert bench.BWD_NAMES == ["chunk_states", "passes", "bwd_chunk", "bwd_dt", "bwd_dA"]
    assert set(f) == set(bench.BWD_NAMES)
