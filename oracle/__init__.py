"""CPU oracle for MLA decode over a latent KV cache.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, calls, links or runs
this package; only the tests, the smoke check and the benchmark's CPU-baseline
leg do. It shares no code, header, table or helper with the CUDA path.

What it computes, and the passages it follows:

* Absorbed MLA attention (``attention.absorbed``): scores against the cached
  latent plus shared rope key, softmax, latent-space output, up-projection
  through W_UV. "GLM-5.2 speculative drafting ... + opt-in MLA-latent KV cache",
  TL;DR item 2 (the DeepSeek "absorb" caches the kv-latent + shared rope key and
  runs attention in latent space).
* Non-absorbed form (``attention.full_head``): per-head K/V decompressed through
  W_UK / W_UV and standard attention, the form the same TL;DR item says the
  absorb was proven equal to (errors ~1e-13).
* Cache footprint (``layout.footprint_elems``): kv_lora_rank + qk_rope_head_dim
  (+ index_head_dim) per token per latent layer, "hf: size GLM-5.3-Flash's KV
  cache from its latent layers only" (#64), PR description.
* Paged layout writer/reader (``layout``).
* Rotation fit, clip thresholds and grouped INT2 codes (``calibrate``,
  ``int2``): "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
  maintainer reply, "How the rotation adapts to the latent": Sigma = c^T c over
  calibration tokens, eigh, eigenvectors in ascending eigenvalue order, clip
  thresholds fit on the rotated latent, attention on the dequantised latent.

Precision: fp64 for all attention arithmetic. The INT2 encoder follows the
fp32 operation order of the encoding definition (plain C, ``int2_quant.c``),
because an integer code is decided there and both sides must decide it in the
same precision.
"""
