"""Plain, slow, fp64 CPU oracle of the calibration-free MoE channel reader.

TEST INFRASTRUCTURE ONLY.  This package is imported, called or executed by
``tests/``, by ``__graft_entry__.smoke()`` and by the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` -- nothing else.  The product path
(the CUDA library and its Python binding) never imports it and shares no code,
header, table or constant generator with it.

Sources (two summaries of the same paper, "Channel Selection for
Mixture-of-Experts Decoding Needs No Calibration Data", Kim & Hwang):

* [CN]  "无需校准数据的MoE解码通道选择 Channel Selection for Mixture-of-Experts
  Decoding Needs No Calibration Data" (Chinese summary page); sections
  前置知识 (background), 核心方法 (core method), 方法步骤详情 (step details).
* [KR]  "MoE 채널 선택은 캘리브레이션 없이 top-k로 충분하다" (Korean summary
  page); sections 어떻게 쓰나 (how to use), 전제와 한계 (assumptions/limits).

Modules
-------
``reader``   the method: rotation, ternary sketch, down norms, recovery basis,
             partial screen, output-unit score, exact global top-k, exact
             gathered compute and low-rank recovery.
``sectors``  32-byte-sector read accounting over the documented array layout.
"""

from . import reader, sectors  # noqa: F401
