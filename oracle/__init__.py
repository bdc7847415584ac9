"""CPU oracle for the SVDQuant W4A4 (NVFP4) linear layer and the AWQ W4A16 GEMV,
and for the epilogues fused onto the linear (GELU of an MLP's first linear;
normalization and rotary embedding of a fused QKV projection, ``qkv``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package-level
smoke check and the benchmark's CPU-baseline leg may import or call anything in
this package.  The product library never imports it and shares no code,
tables or constants with it; the two meet only through the seeded input
generators in ``workloads``.

Everything here is plain and slow on purpose: NumPy in float64 (the formats'
own rounding steps written out exactly), pure-Python ``fractions.Fraction``
for brute force on tiny inputs.  Each function cites the passage of the source
pages it follows.  The pages are news articles about "Nunchaku Lite" in
Diffusers; they name the method (SVDQuant: outliers moved from activations to
weights, a 16-bit low-rank branch, a 4-bit residual), the NVFP4 format with
group size 16 and rank 32, and the AWQ W4A16 family with group size 64, but
give no formula.  The concrete rounding rules used below are the layer's fixed
specification; every point the pages leave open is listed with its reading in
the module that takes it.

Source pages (cited by site and section):
  [dothoosh]  dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion
              models" (Persian) -- the fullest text.
  [hamidun-ar] news.hamidun.com/ar, "Nunchaku Lite: 4-bit image generation in
              Diffusers" -- section "What are Nunchaku and SVDQuant".
  [nextgz]    nextgz.net, "Hugging Face brings Nunchaku Lite to Diffusers" --
              section "Why is W4A4 different from weight-only backends?".
  [hamidun-fr] news.hamidun.com/fr, same article as hamidun-ar (French).

Parity status: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against closed forms, exact rational brute force,
round-trips, a full-rank special case and textbook routines.
"""
