"""Plain fp64 CPU oracle for the TurboQuant quantized KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or call it.  It shares no
code, tables or helpers with the CUDA library under
``turboquant_quantized_kv_gb300/``; the two are written independently from the
same written specification (``include/tq.h``) and the pages it cites.

Sources cited in this package (page title + section):

* [P1] issoh.co.jp, "TurboQuantとは？vLLM・Ollama・LM Studioの対応状況と使い方"
  -- §第1段 (random rotation + per-coordinate Lloyd-Max), §第2段 (QJL 1-bit
  residual, `_nc` = norm correction), §プリセット (K/V bit presets),
  §起動コマンド (first/last two layers kept at full precision),
  §llama.cpp本家 (Hadamard rotation of K/V before the cache).
* [P2] ai-navigate-news.com, turboquant-vllm article -- "Results" (3.76x),
  "Bugs Nobody Else Has Found" (fp32 norms).
* [P3] lilting.ch, "HypuraのNVMeストリーミングとTurboQuantのKVキャッシュ量子化"
  -- "QJL: Johnson-Lindenstrauss変換で残差を1ビット補正する" (residual
  e = x - x_hat, z = R e, sign bits, query projected by the same R, score =
  stage-1 term + QJL correction, R shared by all layers/heads), and the
  KV-size formula section "KVキャッシュ圧縮が実際にボトルネックになるシナリオ".
* [P4] qiita.com, AMD mixed BF16/4-bit KV in LMCache -- "小さな保存・復元コード
  で、責任範囲を確かめる" (4-bit pack `codes[i] | codes[i+1] << 4`, fp32 scale
  appended, 0xA5 guard bytes) and "バイトが同じなら、何が保証されるのか"
  (T(Q(X)) = Q(X)).

Parity status of every function is stated in its module docstring; every
function here is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``.
"""


