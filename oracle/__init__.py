"""fp64 CPU oracle for the rolling-KV step (test infrastructure only).

What it computes is the plain definition the rolling cache is meant to reach
exactly: full-history causal attention under a sliding-window mask, with RoPE
at absolute positions, for single-query decoder steps and for the audio
encoder's incremental multi-query step.  Re-basing and offset bookkeeping are
meant to change nothing (Audio8 ASR Infinite 无限长转写原理, "Rolling KV Cache
三步拆解", 第 2 步: the re-base is an exact rotation; voxtral.c rolling-KV
article, §二 "RoPE 逻辑位置修正": logical position = physical index +
kv_pos_offset), so the oracle never re-bases: it evaluates the definition.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import or run anything in this package.  It shares no
code with the CUDA library and imports nothing from it; the only common
dependency is the seeded input generator in ``synth/``.

Modules
-------
pi         pi from Machin's arctangent formula, exact rational
clock      audio clock / window / delay-token arithmetic of the model card
rope       RoPE frequencies, exact angle reduction, half-split rotation
attention  windowed attention: vectorised definition and explicit-loop brute force
ring       integer model of the per-stream ring state, and the voxtral-style
           compaction it replaces
schemes    fp64 mirrors of the offset-only and exact re-base storage schemes
"""
