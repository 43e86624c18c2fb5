"""Seeded synthetic inputs for the paged decode step.

This module only draws numbers: sequence lengths, the initial order of the
free-block queue, sharing structure and N(0, 1) fp16 tensors.  It holds none
of the paged-attention arithmetic (no block tables, no slots, no softmax);
block tables and slots come from a block manager, and both the CUDA path and
the CPU oracle take their inputs from here.

Workload shapes (OPT-13B attention layer: 40 heads x head_dim 128, fp16,
block size 16; 800 KB of K/V per token over 40 layers -- PagedAttention
notes, unpurerationalist.github.io, §2 "Large KV cache"; default block size
16 -- vLLM paper review, mz-moonzoo.tistory.com/116, §7-2):

* ``tiny``             block 4, pool of 6 blocks, 2 sequences with 9 and 6
                       tokens after the step, 2 heads x 8, one decode step;
* ``opt13b_b64``       64 sequences, context uniform in [128, 2048];
* ``parallel_sampling`` 16 prompts (lognormal, median 160, cap 1024) x 4
                       samples sharing the prompt blocks, 64 decode steps;
* ``mixed_b256``       256 sequences, prompt lognormal (median 200, cap 1536)
                       plus a point inside a lognormal output (median 250),
                       context capped at 2048;
* ``full_40l``         40 layers over a pool-filling cache, context uniform
                       in [512, 2048], optional beam groups of 4 sharing 55 %
                       of their blocks;
* ``prefill_b256``     the prompt phase of the mixed batch: 256 prompts,
                       lognormal (median 200, cap 1536), each prefilled whole.

Readings where the workload text is silent: lognormal sigma = 1.0 with
mu = ln(median), lengths clipped to [1, cap]; a context length counts the
token written in this step, so a sequence holds ``ctx - 1`` tokens before the
step; the pool's free queue starts as a seeded random permutation of its
block ids, so that block tables are fragmented across the pool.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

OPT13B_HEADS = 40
OPT13B_HEAD_DIM = 128
OPT13B_LAYERS = 40
DEFAULT_BLOCK = 16
CTX_CAP = 2048


@dataclass
class DecodeWorkload:
    """Shape and seeded structure of one decode-step workload."""

    name: str
    seed: int
    num_heads: int
    head_dim: int
    block_size: int
    num_layers: int
    num_blocks: int                    # pool size (physical blocks)
    free_order: np.ndarray             # int32 permutation of range(num_blocks)
    prompt_lens: list                  # tokens held by each root sequence before decoding
    # (root_index, number of extra samples forked from it); empty = no sharing
    forks: list = field(default_factory=list)
    # number of leading tokens of each root that are shared before the fork
    # (only used by the beam variant, where beams diverge after a shared prefix)
    shared_prefix: list = field(default_factory=list)
    decode_steps: int = 1
    split_tokens: int = 512            # context partition of the split path
    # total length at which each root sequence finishes (steady-state runs)
    targets: list = field(default_factory=list)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))

    def kv_bytes_per_token(self) -> int:
        return 2 * self.num_heads * self.head_dim * 2


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_f16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) samples rounded to fp16."""
    return rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)


def _lognormal_lengths(rng, n, median, cap, sigma=1.0):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), 1, cap).astype(np.int64)


def _free_order(rng, num_blocks):
    return rng.permutation(num_blocks).astype(np.int32)


def _blocks(n_tokens, block):
    return -(-int(n_tokens) // block)


def tiny(seed: int = 106) -> DecodeWorkload:
    rng = _rng(seed)
    ctx = [9, 6]
    return DecodeWorkload(
        name="tiny", seed=seed, num_heads=2, head_dim=8, block_size=4, num_layers=1,
        num_blocks=6, free_order=_free_order(rng, 6),
        prompt_lens=[c - 1 for c in ctx],
    )


def opt13b_b64(seed: int = 107, batch: int = 64) -> DecodeWorkload:
    rng = _rng(seed)
    ctx = rng.integers(128, CTX_CAP, size=batch, endpoint=True)
    need = sum(_blocks(c, DEFAULT_BLOCK) for c in ctx)
    nb = int(math.ceil(1.25 * need))
    return DecodeWorkload(
        name="opt13b_b64", seed=seed, num_heads=OPT13B_HEADS, head_dim=OPT13B_HEAD_DIM,
        block_size=DEFAULT_BLOCK, num_layers=1, num_blocks=nb,
        free_order=_free_order(rng, nb), prompt_lens=[int(c) - 1 for c in ctx],
    )


def parallel_sampling(seed: int = 108, prompts: int = 16, samples: int = 4,
                      steps: int = 64) -> DecodeWorkload:
    rng = _rng(seed)
    plen = _lognormal_lengths(rng, prompts, 160, 1024)
    need = sum(_blocks(p, DEFAULT_BLOCK) for p in plen)
    # each sample may copy its last block once and grows by `steps` tokens
    need += prompts * samples * (_blocks(steps, DEFAULT_BLOCK) + 2)
    nb = int(math.ceil(1.25 * need))
    return DecodeWorkload(
        name="parallel_sampling", seed=seed, num_heads=OPT13B_HEADS,
        head_dim=OPT13B_HEAD_DIM, block_size=DEFAULT_BLOCK, num_layers=1, num_blocks=nb,
        free_order=_free_order(rng, nb), prompt_lens=[int(p) for p in plen],
        forks=[(i, samples - 1) for i in range(prompts)], decode_steps=steps,
    )


def mixed_b256(seed: int = 109, batch: int = 256, growth_steps: int = 64,
               steady_state: bool = False) -> DecodeWorkload:
    """Mixed-length serving batch.

    Default (a snapshot): each sequence sits at a uniformly drawn point
    1..output of its generation; its target (prompt + output, capped at
    2048) is where it finishes; the pool leaves room for ``growth_steps``
    more tokens per sequence.

    ``steady_state``: the stationary state of a continuous batch that admits
    (prompt, output) pairs from the same distributions -- a slot holds a
    sequence with probability proportional to the steps it stays (target -
    prompt), at a uniform point of its generation -- and a pool with room
    for every sequence at the cap, so replacing finished sequences never
    runs out of blocks.
    """
    rng = _rng(seed)
    if steady_state:
        cand = 64 * batch
        prompt = _lognormal_lengths(rng, cand, 200, 1536)
        target = np.minimum(prompt + _lognormal_lengths(rng, cand, 250, 1 << 30), CTX_CAP)
        stay = (target - prompt).astype(np.float64)
        pick = rng.choice(cand, size=batch, replace=True, p=stay / stay.sum())
        prompt, target = prompt[pick], target[pick]
        done = np.array([rng.integers(1, t - p, endpoint=True) for p, t in zip(prompt, target)],
                        dtype=np.int64)
        ctx = prompt + done
        nb = batch * _blocks(CTX_CAP, DEFAULT_BLOCK)
    else:
        prompt = _lognormal_lengths(rng, batch, 200, 1536)
        output = _lognormal_lengths(rng, batch, 250, 1 << 30)
        done = np.array([rng.integers(1, o, endpoint=True) for o in output], dtype=np.int64)
        ctx = np.minimum(prompt + done, CTX_CAP)
        target = np.minimum(prompt + output, CTX_CAP)
        need = sum(_blocks(c + growth_steps, DEFAULT_BLOCK) for c in ctx)
        nb = int(math.ceil(1.25 * need))
    return DecodeWorkload(
        name="mixed_b256", seed=seed, num_heads=OPT13B_HEADS, head_dim=OPT13B_HEAD_DIM,
        block_size=DEFAULT_BLOCK, num_layers=1, num_blocks=nb,
        free_order=_free_order(rng, nb), prompt_lens=[int(c) - 1 for c in ctx],
        targets=[int(t) for t in target],
    )


def draw_mixed_sequences(rng: np.random.Generator, n: int):
    """``n`` newly admitted sequences of the mixed batch at once:
    (prompt lengths, target lengths), int64 arrays."""
    prompt = _lognormal_lengths(rng, n, 200, 1536)
    output = _lognormal_lengths(rng, n, 250, 1 << 30)
    return prompt, np.minimum(prompt + output, CTX_CAP)


def full_40l(pool_bytes: int, seed: int = 110, beam: bool = False,
             beam_width: int = 4, share: float = 0.55) -> DecodeWorkload:
    """40-layer decode over a pool of ``pool_bytes`` of K/V (all layers).

    Sequences with context uniform in [512, 2048] are admitted until the next
    one would not fit (one block per sequence is kept back for the step's
    growth).  With ``beam``, groups of ``beam_width`` beams share the first
    ``floor(share * blocks)`` whole blocks of their context.
    """
    rng = _rng(seed)
    H, D, B, L = OPT13B_HEADS, OPT13B_HEAD_DIM, DEFAULT_BLOCK, OPT13B_LAYERS
    block_bytes = L * 2 * H * B * D * 2
    nb = int(pool_bytes // block_bytes)
    prompt_lens, forks, shared = [], [], []
    used = 0
    while True:
        ctx = int(rng.integers(512, CTX_CAP, endpoint=True))
        nblk = _blocks(ctx, B)
        if not beam:
            cost = nblk + 1
            if used + cost > nb:
                break
            prompt_lens.append(ctx - 1)
            used += cost
        else:
            pre = int(math.floor(share * nblk))
            own = nblk - pre
            cost = pre + beam_width * (own + 1)
            if used + cost > nb:
                break
            prompt_lens.append(ctx - 1)
            shared.append(pre * B)
            forks.append((len(prompt_lens) - 1, beam_width - 1))
            used += cost
    return DecodeWorkload(
        name="full_40l_beam" if beam else "full_40l", seed=seed, num_heads=H, head_dim=D,
        block_size=B, num_layers=L, num_blocks=nb, free_order=_free_order(rng, nb),
        prompt_lens=prompt_lens, forks=forks, shared_prefix=shared,
    )


WORKLOADS = {
    "tiny": tiny,
    "opt13b_b64": opt13b_b64,
    "parallel_sampling": parallel_sampling,
    "mixed_b256": mixed_b256,
}


def prefill_b256(seed: int = 112, batch: int = 256) -> DecodeWorkload:
    """256 whole prompts drawn like the mixed batch's prompts; the pool holds
    them with 25 % spare blocks and a shuffled free queue."""
    rng = _rng(seed)
    plen = _lognormal_lengths(rng, batch, 200, 1536)
    nb = int(math.ceil(1.25 * sum(_blocks(n, DEFAULT_BLOCK) for n in plen)))
    return DecodeWorkload(name="prefill_b256", seed=seed, num_heads=OPT13B_HEADS,
                          head_dim=OPT13B_HEAD_DIM, block_size=DEFAULT_BLOCK, num_layers=1,
                          num_blocks=nb, free_order=_free_order(rng, nb),
                          prompt_lens=[int(x) for x in plen], decode_steps=0)


def value_rng(workload: DecodeWorkload, stream: int = 0) -> np.random.Generator:
    """Generator for the workload's tensor values (independent of its structure draws)."""
    return _rng(workload.seed * 1000 + 17 + stream)


@dataclass
class BeamChurn:
    """Seeded beam-search churn: ``groups`` requests decode with ``width``
    beams each; after every step each group keeps ``width`` survivors drawn
    (with replacement) from its beams, so a beam drawn m times is kept and
    forked m-1 times and a beam not drawn is freed (PagedAttention notes,
    unpurerationalist.github.io, §3.4.2: beams share ancestor blocks, a
    pruned beam drops its references; vLLM paper review,
    mz-moonzoo.tistory.com/116, §4.4 (2)).  The draws are this generator's;
    applying them to a block manager is the caller's."""

    groups: int
    width: int
    prompt_lens: list
    seed: int

    def survivors(self, rng: np.random.Generator):
        """Per group, the beam indices (0..width-1) kept, with repeats."""
        # beam 0 is likelier: beams of a request tend to collapse onto a few
        p = np.array([2.0] + [1.0] * (self.width - 1))
        return [sorted(rng.choice(self.width, size=self.width, p=p / p.sum()).tolist())
                for _ in range(self.groups)]


def beam_churn(groups: int = 32, width: int = 4, seed: int = 111) -> BeamChurn:
    rng = _rng(seed)
    return BeamChurn(groups=groups, width=width,
                     prompt_lens=[int(x) for x in _lognormal_lengths(rng, groups, 160, 1024)],
                     seed=seed)
