"""CPU oracle for the canvas-denoising hot path -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what one
uniform-state denoising step computes, written in float64 numpy from the
DiffusionGemma explainer ("Understanding DiffusionGemma"): bidirectional
denoising attention and incremental causal prefill ("Architecture:
incremental prefill and denoising"), uniform-state re-noising ("2. Uniform-state
diffusion") and self-conditioning ("Self-conditioning").

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it. The CUDA library never calls it, and it shares no code with the
CUDA library: no kernels, headers, helpers, constants or table generators.
Inputs come from `canvas_denoising_gb300.synth`, which draws random numbers
and holds none of the method's arithmetic.

Every function is pinned by a `-m "not gpu"` test against something other
than itself (numpy's own Philox generator, torch's float64 attention, closed
forms, brute force on tiny inputs); see tests/test_oracle_*.py.
"""
from .philox import philox4x64_10, uniform_token, PHILOX_DOMAIN_RENOISE, PHILOX_DOMAIN_INIT  # noqa: F401
from .attention import canvas_attention  # noqa: F401
from .vocab import vocab_step  # noqa: F401
from .renoise import renoise, canvas_init  # noqa: F401
from .kv import kv_append  # noqa: F401
from .variants import selfcond_input, token_prob, unmask, canvas_fill, finished_early  # noqa: F401
